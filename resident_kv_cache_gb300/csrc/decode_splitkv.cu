// decode_splitkv.cu -- batched single-token decode attention, split-KV, HBM-bound.
//
// Semantics: trueno-gpu 0.4.11 src/memory/resident/attention.rs,
// fn incremental_attention_gpu (one query per head against cache rows
// 0..seq_len-1, zero row for seq_len == 0) and trustformers-core 0.2.0
// src/gpu_ops/cuda/oxicuda/attention.rs, fn attention_decode_gpu_to_gpu (no
// mask), over the batched cache [M, n_kv_heads, max_len, head_dim] of realizar
// 0.8.5 cache_from_cache_from_kv_cache.rs, fn init_batched_kv_cache_gpu.
//
// Design (the pages launch one warp per head, which leaves a 152-SM GPU idle):
//  * A "segment" is the run of valid cache rows of one (sequence m, kv head kh):
//    L_m contiguous rows of D floats.  All segments laid end to end form R rows.
//  * One persistent CTA per SM takes an equal contiguous share of the R rows
//    (balanced to one row whatever the length mix); the share may cross
//    segment boundaries, and each part of a segment in one CTA is a "piece".
//  * A producer warp streams tiles of K and V (8 rows per consumer warp) with bulk
//    async copies into a 2-4 stage shared-memory ring (mbarrier full/empty pairs).
//  * Eleven or twelve consumer warps (eight for G = 8) each take 8 rows of a tile.  GQA: the
//    G = H/Hk query heads that share a kv head are processed together, so every cache row
//    is read from HBM once per kv head.  Dot products are split over the lanes of a row and
//    reduced with a transposing butterfly (one shuffle per partial, not one per
//    head per step); the softmax is online in base 2 with the scale folded into q.
//    For G <= 4 the products and the P.V accumulation run as packed f32x2 FMAs.
//  * Each piece ends with (m, l, o) per head.  A piece that is a whole segment
//    writes the output directly; otherwise it writes a partial record to the
//    workspace, and the last CTA to finish a segment (atomic ticket) merges the
//    records with the log-sum-exp rule, one warp per query head, and resets the
//    ticket to zero.
//  * With k_new / v_new (the one-launch decode step), the new row of a segment is its
//    last row, len-1.  The CTA whose share holds it copies that row into its last tile
//    straight from k_new / v_new (the tile's other rows come from the cache), so no
//    copy of this launch reads cache row len-1, and the consumer warps write the new
//    rows into the cache after their last piece, with nothing waiting on the stores.
#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

constexpr int kDecBatchRows = 8;                                   // rows per warp per tile
constexpr int kDecMaxCtas = 1024;
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int ilog2c(int x) { return x <= 1 ? 0 : 1 + ilog2c(x / 2); }

template <int D, int G>
struct DecCfg {
    // Consumer warps: 11 or 12 hide the shared-memory and shuffle latencies better than 8;
    // G = 8 needs more registers.
    // FPL float4 columns of a row per lane: 2 for D >= 64 at G <= 4 halves the butterfly that
    // sums the partial dot products; the extra q and accumulator registers need the 170 a
    // thread gets with 12 warps per CTA (3 per sub-partition), so 11 consumer warps there.
    static constexpr int FPL = (G <= 4 && D >= 64) ? 2 : 1;
    static constexpr int W = FPL == 2 ? 11 : (G <= 4 ? 12 : 8);
    static constexpr int CT = W * 32;                 // consumer threads
    static constexpr int THREADS = CT + 32;           // + one producer warp
    static constexpr int TILE_ROWS = kDecBatchRows * W;
    static constexpr int D4 = D / 4;                  // float4 per cache row
    static constexpr int LPR = D4 / FPL;              // lanes per cache row
    static constexpr int RPW = 32 / LPR;              // rows a warp covers per pass
    static constexpr int PASSES = kDecBatchRows / RPW;
    static constexpr int NV = PASSES * G;             // partial dot products per lane
    static constexpr int NVR = NV >= LPR ? NV / LPR : 1;   // totals per lane after the butterfly
    static constexpr int ENTRIES = kDecBatchRows * G; // scores per warp per tile
    static constexpr int EPL = ENTRIES >= 32 ? ENTRIES / 32 : 1;
    static constexpr int REC = ((G * D + 2 * G) + 3) / 4 * 4;      // floats per partial record
    // shared memory layout (bytes): as many K/V stages as fit beside the reduction buffers
    static constexpr int TILE_BYTES = TILE_ROWS * D * 4;
    static constexpr int SIDE = W * ENTRIES * 4 + W * G * D * 4 + W * 2 * G * 4 + 34 * 8 + 32 * 4 + 2 * 4 * 8 + 16 +
                                2 * 32 * 8 + 32 * 4;
    static constexpr int NST_FIT = (226 * 1024 - SIDE) / (2 * TILE_BYTES);
    static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;          // pipeline stages
    static_assert(NST >= 2, "decode pipeline needs two stages");
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_SC = OFF_STAGES + NST * 2 * TILE_BYTES;
    static constexpr int OFF_RED_ACC = OFF_SC + W * ENTRIES * 4;
    static constexpr int OFF_RED_ML = OFF_RED_ACC + W * G * D * 4;
    static constexpr int OFF_P = OFF_RED_ML + W * 2 * G * 4;      // int64 P[33]
    static constexpr int OFF_L = OFF_P + 34 * 8;                                  // int L[32]
    static constexpr int OFF_BAR = OFF_L + 32 * 4;                                // full/empty
    static constexpr int OFF_MISC = OFF_BAR + 2 * NST * 8;                        // abort, last
    static constexpr int OFF_PTR = OFF_MISC + 16;                                 // per-sequence K, V bases
    static constexpr int OFF_APP = OFF_PTR + 2 * 32 * 8;                          // int APP[32]
    static constexpr int SMEM = OFF_APP + 32 * 4;
    static_assert(SMEM <= 227 * 1024, "decode shared memory budget");
    static_assert(NV >= 1 && (LPR & (LPR - 1)) == 0, "lane split");
};

// Sum NV per-lane values across W lanes (W a power of two): halving exchanges
// leave each lane the totals of a distinct slice of indices, then plain
// butterflies finish when fewer values than lanes remain.  After it, a lane
// holds v[0..NVR) = totals of indices (lane % W) * (NV / W) + t when NV >= W,
// or v[0] = total of index (lane % W) / (W / NV) when NV < W.
template <int NV, int W>
__device__ __forceinline__ void xpose_reduce(float (&v)[NV], int lane) {
    constexpr int HSTEPS = ilog2c(NV) < ilog2c(W) ? ilog2c(NV) : ilog2c(W);
#pragma unroll
    for (int s = 0; s < HSTEPS; ++s) {
        const int o = (W >> 1) >> s;
        const int half = (NV >> s) >> 1;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    constexpr int C = NV >> HSTEPS;
#pragma unroll
    for (int o = (W >> 1) >> HSTEPS; o >= 1; o >>= 1) {
#pragma unroll
        for (int i = 0; i < C; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    }
}

// Owner CTA of flat row `pos` when R rows are cut into n shares
// [floor(R*c/n), floor(R*(c+1)/n)).
__device__ __forceinline__ int owner_of(int64_t pos, int64_t R, int n) {
    const int64_t c = ((pos + 1) * (int64_t)n - 1) / R;
    return c < n - 1 ? (int)c : n - 1;
}

// First flat row of CTA c's share.
__device__ __forceinline__ int64_t share_begin(int c, int64_t R, int n) { return R * c / n; }

// Segment containing flat row pos: sequence m (P[m] <= pos < P[m+1]) and kv head.
__device__ __forceinline__ void locate(int64_t pos, const int64_t* P, const int* L, int Hk, int& m, int& kh,
                                       int64_t& seg_start) {
    m = 0;
    while (P[m + 1] <= pos) ++m;
    kh = (int)((pos - P[m]) / L[m]);
    seg_start = P[m] + (int64_t)kh * L[m];
    (void)Hk;
}

template <int D, int G>
__global__ void __launch_bounds__(DecCfg<D, G>::THREADS, 1)
decode_splitkv_kernel(const float* __restrict__ q, const float* __restrict__ k_cache,
                      const float* __restrict__ v_cache, const float* const* __restrict__ k_ptrs,
                      const float* const* __restrict__ v_ptrs, float* __restrict__ out, int M, int Hk, int Lmax,
                      const int* __restrict__ seq_lens, float scale_log2, int* __restrict__ tickets,
                      float* __restrict__ records, unsigned int* __restrict__ flags,
                      const float* __restrict__ k_new, const float* __restrict__ v_new) {
    using C = DecCfg<D, G>;
    extern __shared__ __align__(1024) unsigned char smem[];
    float* sc_all = reinterpret_cast<float*>(smem + C::OFF_SC);
    float* red_acc = reinterpret_cast<float*>(smem + C::OFF_RED_ACC);
    float* red_ml = reinterpret_cast<float*>(smem + C::OFF_RED_ML);
    int64_t* P = reinterpret_cast<int64_t*>(smem + C::OFF_P);
    int* L = reinterpret_cast<int*>(smem + C::OFF_L);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    int* APP = reinterpret_cast<int*>(smem + C::OFF_APP);   // [m]: a new row goes to row L[m]-1
    const float** kbase = reinterpret_cast<const float**>(smem + C::OFF_PTR);   // [32]
    const float** vbase = kbase + 32;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n = gridDim.x;
    const int c = blockIdx.x;
    const int H = Hk * G;

    // ---- prologue: lengths, prefix sums, barriers
    if (warp == 0) {
        int len = 0;
        if (lane < M) {
            len = __ldg(seq_lens + lane);
            if (len > Lmax) { len = Lmax; atomicOr(flags, RKV_FLAG_LEN_CLAMPED); }
            if (len < 0) { len = 0; atomicOr(flags, RKV_FLAG_NEGATIVE_INPUT); }
            // the sequence's cache: a slice of the batched cache, or its own allocation (pointer
            // arrays); a null or misaligned base is never read -- the sequence counts as empty
            const float* kb = k_ptrs ? k_ptrs[lane] : k_cache + (int64_t)lane * Hk * Lmax * D;
            const float* vb = v_ptrs ? v_ptrs[lane] : v_cache + (int64_t)lane * Hk * Lmax * D;
            if (!kb || !vb || ((reinterpret_cast<uintptr_t>(kb) | reinterpret_cast<uintptr_t>(vb)) & 15u)) {
                len = 0;
                atomicOr(flags, RKV_FLAG_BAD_POINTER);
            }
            kbase[lane] = kb;
            vbase[lane] = vb;
            L[lane] = len;
            // the step's new row lands at len-1 only for a length in [1, max_len] (unclamped) and a
            // usable cache; it is then the last row of each of the sequence's segments
            APP[lane] = k_new != nullptr && len > 0 && len == __ldg(seq_lens + lane);
        }
        int64_t rows = (int64_t)len * Hk, incl = rows;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane < M) P[lane + 1] = incl;
        if (lane == 0) { P[0] = 0; *abort_flag = 0; *last_flag = 0; }
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);                          // full: producer arrival + tx
            mbar_init(smem_addr(&bars[C::NST + s]), C::W);  // empty: one per consumer warp
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t R = P[M];
    const int64_t r0 = share_begin(c, R, n), r1 = share_begin(c + 1, R, n);

    if (warp == C::W) {
        // ================================================================ producer
        if (lane == 0) {
            int issued[C::NST > 0 ? C::NST : 1];
            for (int s = 0; s < C::NST; ++s) issued[s] = 0;
            int it = 0;
            bool ok = true;
            int64_t pos = r0;
            // K/V rows are read once per step: evict-first in L2, so the stream does not push
            // out (and force the write-back of) lines other kernels left dirty.
            const uint64_t stream_policy = l2_policy_evict_first();
            while (ok && pos < r1) {
                int m, kh;
                int64_t seg_start;
                locate(pos, P, L, Hk, m, kh, seg_start);
                const int64_t piece_end = min(r1, seg_start + L[m]);
                const int64_t head_row0 = (int64_t)kh * Lmax - seg_start;  // flat -> row of the sequence's cache
                const float* kb = kbase[m];
                const float* vb = vbase[m];
                for (int64_t t0 = pos; t0 < piece_end; t0 += C::TILE_ROWS, ++it) {
                    const int s = it % C::NST;
                    const uint32_t ph = (uint32_t)(it / C::NST) & 1u;
                    if (!mbar_wait(smem_addr(&bars[C::NST + s]), ph ^ 1u, abort_flag, flags)) { ok = false; break; }
                    const int rows = (int)min((int64_t)C::TILE_ROWS, piece_end - t0);
                    // the tile that ends a segment with a new row takes that row from k_new / v_new
                    const bool new_row = APP[m] && t0 + rows == seg_start + L[m];
                    const int cache_rows = rows - (new_row ? 1 : 0);
                    const uint32_t bytes = (uint32_t)cache_rows * D * 4;
                    const uint32_t full = smem_addr(&bars[s]);
                    const uint32_t k_dst = smem_addr(smem + C::OFF_STAGES + (2 * s) * C::TILE_BYTES);
                    const uint32_t v_dst = smem_addr(smem + C::OFF_STAGES + (2 * s + 1) * C::TILE_BYTES);
                    // (checked build) rows of this sequence's cache, and its row of k_new / v_new
                    if (!in_bounds(head_row0 + t0, (int64_t)Hk * Lmax, flags) ||
                        !in_bounds(head_row0 + t0 + rows - 1, (int64_t)Hk * Lmax, flags) ||
                        !in_bounds((int64_t)m * Hk + kh, (int64_t)M * Hk, flags)) {
                        mbar_arrive(full);        // no copy: the consumers see stale rows, the flag says so
                        issued[s] = it + 1;
                        continue;
                    }
                    mbar_arrive_expect_tx(full, 2u * (uint32_t)rows * D * 4);
                    const int64_t src = (head_row0 + t0) * D;
                    if (cache_rows > 0) {
                        bulk_g2s_hint(k_dst, kb + src, bytes, full, stream_policy);
                        bulk_g2s_hint(v_dst, vb + src, bytes, full, stream_policy);
                    }
                    if (new_row) {
                        const int64_t nr = ((int64_t)m * Hk + kh) * D;
                        bulk_g2s_hint(k_dst + bytes, k_new + nr, D * 4, full, stream_policy);
                        bulk_g2s_hint(v_dst + bytes, v_new + nr, D * 4, full, stream_policy);
                    }
                    issued[s] = it + 1;
                }
                pos = piece_end;
            }
            if (!ok) {   // unwinding: let copies already issued land before the CTA exits
                for (int s = 0; s < C::NST; ++s)
                    if (issued[s] > 0)
                        mbar_drain(smem_addr(&bars[s]), (uint32_t)((issued[s] - 1) / C::NST) & 1u, 100000000ull);
            }
        }
        return;
    }

    // ==================================================================== consumers
    // Zero rows for empty sequences (no rows in the partition covers them).
    for (int sg = c; sg < M * Hk; sg += n) {
        const int m = sg / Hk, kh = sg % Hk;
        if (L[m] == 0)
            for (int i = threadIdx.x; i < G * D; i += C::CT)
                if (in_bounds((int64_t)m * H * D + (int64_t)(kh * G) * D + i, (int64_t)M * H * D, flags))
                    out[(int64_t)m * H * D + (int64_t)(kh * G) * D + i] = 0.0f;
    }

    const int seg = lane % C::LPR;         // float4 column of this lane
    const int rgrp = lane / C::LPR;        // row group within a pass
    float* sc = sc_all + warp * C::ENTRIES;

    float4 qv[G][C::FPL];
    float acc[G][4 * C::FPL];
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    int it = 0;
    int64_t pos = r0;
    while (pos < r1) {
        int m, kh;
        int64_t seg_start;
        locate(pos, P, L, Hk, m, kh, seg_start);
        const int64_t seg_end = seg_start + L[m];
        const int64_t piece_end = min(r1, seg_end);
        // q of the G heads sharing kv head kh, pre-scaled so scores are in log2 units
        const bool q_ok = in_bounds((int64_t)m * H * D + (int64_t)(kh * G + G) * D - 1, (int64_t)M * H * D, flags);
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int f = 0; f < C::FPL; ++f) {
                float4 t = q_ok ? __ldg(reinterpret_cast<const float4*>(q + (int64_t)m * H * D + (int64_t)(kh * G + h) * D) +
                                        seg + f * C::LPR)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                qv[h][f] = make_float4(t.x * scale_log2, t.y * scale_log2, t.z * scale_log2, t.w * scale_log2);
            }
#pragma unroll
            for (int j = 0; j < 4 * C::FPL; ++j) acc[h][j] = 0.0f;
        }
        m_run = -INFINITY;
        l_run = 0.0f;

        for (int64_t t0 = pos; t0 < piece_end; t0 += C::TILE_ROWS, ++it) {
            const int s = it % C::NST;
            const uint32_t ph = (uint32_t)(it / C::NST) & 1u;
            if (ok) ok = mbar_wait(smem_addr(&bars[s]), ph, abort_flag, flags);
            const int tile_rows = (int)min((int64_t)C::TILE_ROWS, piece_end - t0);
            const int nvalid = min(max(tile_rows - warp * kDecBatchRows, 0), kDecBatchRows);
            if (ok && nvalid > 0) {
                const float4* Ks = reinterpret_cast<const float4*>(smem + C::OFF_STAGES + (2 * s) * C::TILE_BYTES) +
                                   (warp * kDecBatchRows) * C::D4;
                const float4* Vs = reinterpret_cast<const float4*>(smem + C::OFF_STAGES + (2 * s + 1) * C::TILE_BYTES) +
                                   (warp * kDecBatchRows) * C::D4;
                // ---- partial dot products: pass p covers rows p*RPW .. p*RPW+RPW-1
                float part[C::NV];
#pragma unroll
                for (int p = 0; p < C::PASSES; ++p) {
                    const int row = p * C::RPW + rgrp;
                    float4 kv[C::FPL];
#pragma unroll
                    for (int f = 0; f < C::FPL; ++f)
                        kv[f] = row < nvalid ? Ks[row * C::D4 + seg + f * C::LPR] : make_float4(0.f, 0.f, 0.f, 0.f);
                    if constexpr (G <= 4) {
                        // q.k of the lane's dims as packed f32x2 products (x,y and z,w lanes) summed;
                        // at G = 8 the packed form needs more registers than it saves
#pragma unroll
                        for (int h = 0; h < G; ++h) {
                            uint64_t t = f2_mul(f2_pack(qv[h][0].x, qv[h][0].y), f2_pack(kv[0].x, kv[0].y));
                            t = f2_fma(f2_pack(qv[h][0].z, qv[h][0].w), f2_pack(kv[0].z, kv[0].w), t);
#pragma unroll
                            for (int f = 1; f < C::FPL; ++f) {
                                t = f2_fma(f2_pack(qv[h][f].x, qv[h][f].y), f2_pack(kv[f].x, kv[f].y), t);
                                t = f2_fma(f2_pack(qv[h][f].z, qv[h][f].w), f2_pack(kv[f].z, kv[f].w), t);
                            }
                            float a, b;
                            f2_unpack(t, a, b);
                            part[p * G + h] = a + b;
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < G; ++h) {
                            float t = 0.0f;
#pragma unroll
                            for (int f = 0; f < C::FPL; ++f)
                                t += qv[h][f].x * kv[f].x + qv[h][f].y * kv[f].y + qv[h][f].z * kv[f].z +
                                     qv[h][f].w * kv[f].w;
                            part[p * G + h] = t;
                        }
                    }
                }
                xpose_reduce<C::NV, C::LPR>(part, lane);
                // ---- scatter the totals to sc[row * G + h]
#pragma unroll
                for (int t = 0; t < C::NVR; ++t) {
                    int idx;
                    bool writer;
                    if (C::NV >= C::LPR) {
                        idx = seg * (C::NV / C::LPR) + t;
                        writer = true;
                    } else {
                        constexpr int dup = (C::NV >= C::LPR) ? 1 : C::LPR / C::NV;
                        idx = seg / dup;
                        writer = (seg % dup) == 0;
                    }
                    const int p = idx / G, h = idx % G;
                    const int row = p * C::RPW + rgrp;
                    if (writer) sc[row * G + h] = part[t];
                }
                __syncwarp();
                // ---- online softmax over this batch (base 2)
                float sv[C::EPL];
                float bmax = -INFINITY;
#pragma unroll
                for (int k = 0; k < C::EPL; ++k) {
                    const int e = lane + 32 * k;
                    const bool valid = e < C::ENTRIES && (e / G) < nvalid;
                    sv[k] = valid ? sc[e] : -INFINITY;
                    bmax = fmaxf(bmax, sv[k]);
                }
#pragma unroll
                for (int o = G; o < 32; o <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
                const float m_new = fmaxf(m_run, bmax);
                const float alpha = (m_new == -INFINITY) ? 1.0f : fast_exp2(m_run - m_new);
                float bsum = 0.0f;
#pragma unroll
                for (int k = 0; k < C::EPL; ++k) {
                    const int e = lane + 32 * k;
                    const float p = (sv[k] == -INFINITY) ? 0.0f : fast_exp2(sv[k] - m_new);
                    bsum += p;
                    if (e < C::ENTRIES) sc[e] = p;
                }
#pragma unroll
                for (int o = G; o < 32; o <<= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, o);
                l_run = l_run * alpha + bsum;
                m_run = m_new;
                __syncwarp();
                // ---- rescale and accumulate P.V
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float a = __shfl_sync(0xffffffffu, alpha, h);
                    if constexpr (G <= 4) {
                        const uint64_t a2 = f2_pack(a, a);
#pragma unroll
                        for (int j = 0; j < 4 * C::FPL; j += 2)
                            f2_unpack(f2_mul(f2_pack(acc[h][j], acc[h][j + 1]), a2), acc[h][j], acc[h][j + 1]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4 * C::FPL; ++j) acc[h][j] *= a;
                    }
                }
#pragma unroll
                for (int p = 0; p < C::PASSES; ++p) {
                    const int row = p * C::RPW + rgrp;
                    if (row < nvalid) {
                        float4 vv[C::FPL];
#pragma unroll
                        for (int f = 0; f < C::FPL; ++f) vv[f] = Vs[row * C::D4 + seg + f * C::LPR];
                        if constexpr (G <= 4) {
                            // acc += w * v, two dims per packed f32x2 FMA (per-lane rounding as fmaf)
#pragma unroll
                            for (int h = 0; h < G; ++h) {
                                const float w = sc[row * G + h];
                                const uint64_t w2 = f2_pack(w, w);
#pragma unroll
                                for (int f = 0; f < C::FPL; ++f) {
                                    float* a4 = acc[h] + 4 * f;
                                    f2_unpack(f2_fma(w2, f2_pack(vv[f].x, vv[f].y), f2_pack(a4[0], a4[1])), a4[0], a4[1]);
                                    f2_unpack(f2_fma(w2, f2_pack(vv[f].z, vv[f].w), f2_pack(a4[2], a4[3])), a4[2], a4[3]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int h = 0; h < G; ++h) {
                                const float w = sc[row * G + h];
#pragma unroll
                                for (int f = 0; f < C::FPL; ++f) {
                                    acc[h][4 * f + 0] += w * vv[f].x;
                                    acc[h][4 * f + 1] += w * vv[f].y;
                                    acc[h][4 * f + 2] += w * vv[f].z;
                                    acc[h][4 * f + 3] += w * vv[f].w;
                                }
                            }
                        }
                    }
                }
            }
            if (ok && *abort_flag) ok = false;
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(smem_addr(&bars[C::NST + s]));
        }

        // ---------------------------------------------------------- piece end
        // rows of different row groups share the warp's running max: plain sums
#pragma unroll
        for (int o = C::LPR; o < 32; o <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int j = 0; j < 4 * C::FPL; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], o);
        if (lane < C::LPR) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int f = 0; f < C::FPL; ++f)
                    *reinterpret_cast<float4*>(red_acc + (warp * G + h) * D + (seg + f * C::LPR) * 4) =
                        make_float4(acc[h][4 * f], acc[h][4 * f + 1], acc[h][4 * f + 2], acc[h][4 * f + 3]);
        }
        if (lane < G) {
            red_ml[(warp * G + lane) * 2 + 0] = m_run;
            red_ml[(warp * G + lane) * 2 + 1] = l_run;
        }
        named_barrier(1, C::CT);

        const int sg = m * Hk + kh;
        const int c_first = owner_of(seg_start, R, n);
        const int c_last = owner_of(seg_end - 1, R, n);
        const bool single = (c_first == c_last);
        float* my_rec = records + (int64_t)(sg + c) * C::REC;
        float* o_seg = out + (int64_t)m * H * D + (int64_t)(kh * G) * D;
        // (checked build) this piece's record, its segment's ticket and output rows
        const bool io_ok = in_bounds((int64_t)sg + c, (int64_t)M * Hk + kDecMaxCtas, flags) &&
                           in_bounds(sg, kDecodeTicketSlots, flags) &&
                           in_bounds((int64_t)m * H * D + (int64_t)(kh * G) * D + G * D - 1, (int64_t)M * H * D, flags);
        for (int i = threadIdx.x; i < G * D; i += C::CT) {
            const int h = i / D, d = i % D;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::W; ++w) mx = fmaxf(mx, red_ml[(w * G + h) * 2]);
            float l = 0.0f, o = 0.0f;
            if (mx != -INFINITY) {
#pragma unroll
                for (int w = 0; w < C::W; ++w) {
                    const float mw = red_ml[(w * G + h) * 2];
                    const float f = (mw == -INFINITY) ? 0.0f : fast_exp2(mw - mx);
                    l += red_ml[(w * G + h) * 2 + 1] * f;
                    o += red_acc[(w * G + h) * D + d] * f;
                }
            }
            if (!io_ok) {
                // skipped
            } else if (single) {
                o_seg[i] = l > 0.0f ? o / l : 0.0f;
            } else {
                my_rec[i] = o;
                if (d == 0) {
                    my_rec[G * D + h] = mx;
                    my_rec[G * D + G + h] = l;
                }
            }
        }
        if (!single) {
            __threadfence();
            named_barrier(1, C::CT);
            if (threadIdx.x == 0) {
                // pieces = CTAs in [c_first, c_last] that own rows (a share is empty only when R < n)
                int pieces = c_last - c_first + 1;
                if (R < n) {
                    pieces = 0;
                    for (int cc = c_first; cc <= c_last; ++cc)
                        pieces += share_begin(cc, R, n) < share_begin(cc + 1, R, n);
                }
                int last = 0;
                if (ok && io_ok) last = (atomicAdd(tickets + sg, 1) == pieces - 1);
                *last_flag = last;
            }
            named_barrier(1, C::CT);
            if (*last_flag) {
                // Log-sum-exp merge of the segment's records, one warp per query head: the lanes
                // find the largest running max together, then walk the records once -- m and l
                // are the same address for every lane (one broadcast load), each lane takes a
                // float4 of o -- four records at a time so their loads overlap.
                __threadfence();
                const bool all_owned = R >= n;          // then every CTA in [c_first, c_last] has a record
                for (int h = warp; h < G; h += C::W) {
                    float mx = -INFINITY;
                    for (int cc = c_first + lane; cc <= c_last; cc += 32)
                        if (all_owned || share_begin(cc, R, n) < share_begin(cc + 1, R, n))
                            mx = fmaxf(mx, __ldcg(records + (int64_t)(sg + cc) * C::REC + G * D + h));
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    float l = 0.0f;
                    float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    const bool has_col = lane < D / 4;
                    if (mx != -INFINITY) {
#pragma unroll 4
                        for (int cc = c_first; cc <= c_last; ++cc) {
                            if (!all_owned && !(share_begin(cc, R, n) < share_begin(cc + 1, R, n))) continue;
                            const float* rec = records + (int64_t)(sg + cc) * C::REC;
                            const float mc = __ldcg(rec + G * D + h);
                            const float lc = __ldcg(rec + G * D + G + h);
                            const float4 oc = has_col ? __ldcg(reinterpret_cast<const float4*>(rec + h * D) + lane)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                            const float f = (mc == -INFINITY) ? 0.0f : fast_exp2(mc - mx);
                            l += lc * f;
                            o4.x += oc.x * f;
                            o4.y += oc.y * f;
                            o4.z += oc.z * f;
                            o4.w += oc.w * f;
                        }
                    }
                    if (has_col) {
                        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                        reinterpret_cast<float4*>(o_seg + h * D)[lane] =
                            make_float4(o4.x * inv, o4.y * inv, o4.z * inv, o4.w * inv);
                    }
                }
                if (threadIdx.x == 0) tickets[sg] = 0;
            }
        }
        named_barrier(1, C::CT);   // red_* free for the next piece
        pos = piece_end;
    }
    if (k_new) {
        // The step's new rows into the cache, for the segments whose last row is in this CTA's
        // share.  No copy of this launch reads those rows (their tiles took them from k_new /
        // v_new), so the stores wait for nothing and nothing waits for them.
        for (int sg = warp; sg < M * Hk; sg += C::W) {
            const int m = sg / Hk, kh = sg - m * Hk;
            if (!APP[m]) continue;
            const int64_t flat = P[m] + (int64_t)(kh + 1) * L[m] - 1;
            if (flat < r0 || flat >= r1) continue;
            const int64_t row = ((int64_t)kh * Lmax + L[m] - 1) * D;
            const int64_t nr = ((int64_t)m * Hk + kh) * D;
            if (!in_bounds(row + D - 1, (int64_t)Hk * Lmax * D, flags) || !in_bounds(nr + D - 1, (int64_t)M * Hk * D, flags))
                continue;
            for (int i = lane; i < D / 4; i += 32) {
                reinterpret_cast<float4*>(const_cast<float*>(kbase[m]) + row)[i] =
                    __ldg(reinterpret_cast<const float4*>(k_new + nr) + i);
                reinterpret_cast<float4*>(const_cast<float*>(vbase[m]) + row)[i] =
                    __ldg(reinterpret_cast<const float4*>(v_new + nr) + i);
            }
        }
    }
}

// ------------------------------------------------------------------ host side
bool decode_group_supported(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

template <int D, int G>
static constexpr int rec_floats() { return DecCfg<D, G>::REC; }

static int rec_floats_rt(int D, int G) {
    return ((G * D + 2 * G) + 3) / 4 * 4;
}

size_t decode_workspace_bytes(int M, int H, int Hk, int D) {
    const int G = H / Hk;
    return (size_t)RKV_DECODE_TICKET_BYTES + (size_t)(M * Hk + kDecMaxCtas) * rec_floats_rt(D, G) * 4;
}

template <int D, int G>
static rkv_status launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
    using C = DecCfg<D, G>;
    static_assert(rec_floats<D, G>() == ((G * D + 2 * G) + 3) / 4 * 4, "record layout");
    auto kern = decode_splitkv_kernel<D, G>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return check_launch("attn_decode_batched: shared-memory attribute");
        attr_done[dev] = true;
    }
    int n = sm_count();
    if (n <= 0) return set_error(RKV_ERR_LAUNCH, "attn_decode_batched: cannot query the SM count");
    if (n > kDecMaxCtas) n = kDecMaxCtas;
    int* tickets = static_cast<int*>(a.workspace);
    float* records = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + RKV_DECODE_TICKET_BYTES);
    kern<<<n, C::THREADS, C::SMEM, stream>>>(a.q, a.k_cache, a.v_cache, a.k_ptrs, a.v_ptrs, a.o, a.M, a.Hk, a.Lmax,
                                               a.seq_lens, a.scale * kLog2e, tickets, records, a.flags, a.k_new,
                                               a.v_new);
    return check_launch("attn_decode_batched");
}

rkv_status launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    const int G = a.H / a.Hk;
#define RKV_DEC_CASE(DD, GG) \
    if (a.D == DD && G == GG) return launch_decode_t<DD, GG>(a, stream);
    RKV_DEC_CASE(16, 1) RKV_DEC_CASE(16, 2) RKV_DEC_CASE(16, 4) RKV_DEC_CASE(16, 8)
    RKV_DEC_CASE(32, 1) RKV_DEC_CASE(32, 2) RKV_DEC_CASE(32, 4) RKV_DEC_CASE(32, 8)
    RKV_DEC_CASE(64, 1) RKV_DEC_CASE(64, 2) RKV_DEC_CASE(64, 4) RKV_DEC_CASE(64, 8)
    RKV_DEC_CASE(128, 1) RKV_DEC_CASE(128, 2) RKV_DEC_CASE(128, 4) RKV_DEC_CASE(128, 8)
#undef RKV_DEC_CASE
    return set_error(RKV_ERR_UNSUPPORTED, "attn_decode_batched: head_dim %d with group %d", a.D, G);
}

}  // namespace rkv
