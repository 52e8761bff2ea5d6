// prefill_tc.cu -- fused flash-style prefill on the 5th-generation tensor core (sm_103a).
//
// Semantics: trueno-gpu 0.4.11 src/memory/resident/attention.rs,
// fn batched_multihead_attention_optimized (interleaved [seq, n_heads*head_dim]
// in and out, scale 1/sqrt(head_dim)) and trustformers-core 0.2.0
// src/gpu_ops/cuda/oxicuda/attention.rs, fn attention_prefill_gpu_to_gpu
// (causal: query i sees keys 0..=i; per head: scaled GEMM, causal softmax,
// GEMM).  Here all of it is one kernel: heads are read in place, the score
// tile never leaves tensor memory, and softmax is online (base 2).
//
// One CTA computes a 128-query tile of one (batch, head):
//   warp 0       K producer: TMA (cp.async.bulk.tensor, 128-byte swizzle) of
//                BN x D key tiles into an NK-stage ring, K-major for the MMA.
//   warp 1       MMA issuer (one thread) and TMEM owner:
//                  S_j  = Q . K_j^T   tcgen05.mma kind::tf32, A = Q from TMEM
//                  O   += P_j . V_j   tcgen05.mma kind::tf32, A = P from TMEM
//                S is double-buffered in TMEM so QK^T of block j+1 overlaps the
//                softmax of block j.
//   warps 2-5    softmax / epilogue, one thread per query row (TMEM lane):
//                Q rows -> TMEM (pre-scaled by scale*log2e, rounded to TF32),
//                then per block: S row from TMEM, mask, row max, lazy rescale
//                (O is rescaled only when the running max grows by more than
//                2^8), p = 2^(s - m) rounded to TF32 and written back over S,
//                then O / l stored to the interleaved output row.
//   warps 6-9    V transposer: tcgen05 kind::tf32 reads B only K-major, so V
//                tiles are loaded with 16-byte loads, transposed in registers
//                (4x4 blocks), rounded to TF32 and stored K-major (128-byte
//                swizzle, conflict-free 16-byte stores) into an NV-stage ring.
// Every mbarrier wait is time-bounded (see rkv_internal.cuh); a CTA that gives
// up unwinds: it drains its own copies in flight, lets issued MMAs finish and
// frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

constexpr int kPfBM = 128;                    // query rows per CTA (TMEM lanes)
constexpr int kPfThreads = 352;               // 11 warps
constexpr int kPfPvWarp = 10;                 // PV issuer
constexpr int kPfSoftmaxWarp0 = 2;
constexpr int kPfVWarp0 = 6;
constexpr uint32_t kPfTmemCols = 512;
constexpr uint32_t kColQ = 0, kColO = 128, kColS = 256;   // TMEM column bases
constexpr float kPfLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.0f;          // log2 of the largest unnormalised p kept
constexpr int kPfMinSmem = 120 * 1024;        // keeps one CTA per SM (TMEM is allocated whole)

template <int D>
struct PfCfg {
    static constexpr int BN = D == 128 ? 64 : 128;          // keys per block
    static constexpr int CH = D >= 32 ? 32 : D;             // floats per swizzled K row chunk
    static constexpr int NCH = D / CH;
    static constexpr int TILE = BN * D * 4;                 // bytes of one K or V^T tile
    // D = 128: K slots come in adjacent pairs so one N = 128 MMA chain computes the scores
    // of two 64-key blocks (half the MMAs of N = 64; a thread needs ~45+ cycles per issue).
    static constexpr bool KPAIR = D == 128;
    static constexpr int NK = KPAIR ? 4 : (D >= 64 ? 3 : 4);   // K stages
    static constexpr int NV = D >= 64 ? 3 : 4;              // V^T stages
    // S/P buffers in TMEM: the MMA issuer runs up to NSBUF blocks of QK^T ahead of the
    // softmax, so the tensor core always has queued work.  D <= 64: PV is split over
    // even/odd key steps into two accumulators (O = O_a + O_b).
    static constexpr int NSBUF = D == 128 ? 4 : 2;
    static constexpr int PV_SPLIT = D <= 64 ? 2 : 1;
    static constexpr int S_BUF = BN;                       // TMEM columns of one S buffer
    static constexpr uint32_t K_SWIZZLE = D >= 32 ? kSwizzle128B : kSwizzle64B;
    // Q arrives by TMA into V ring slots 1 .. QSLOTS (free until V blocks 1.. are loaded)
    static constexpr int QSLOTS = kPfBM / BN;
    static_assert(1 + QSLOTS <= NV, "Q staging slots");
    static constexpr uint32_t K_ATOM = D >= 32 ? 1024 : 512; // 8 rows x swizzle span
    // shared memory layout (offsets from a 1024-aligned base)
    static constexpr int OFF_K = 0;
    // byte offset of d-chunk c of K slot s: paired slots interleave their chunks so the
    // 2*BN rows of a chunk are contiguous (uniform 1024-byte stride per 8 rows)
    __host__ __device__ static constexpr int koff(int s, int c) {
        return KPAIR ? (s / 2) * 2 * TILE + c * (2 * BN * CH * 4) + (s % 2) * (BN * CH * 4)
                     : s * TILE + c * (BN * CH * 4);
    }
    static constexpr int OFF_V = OFF_K + NK * TILE;
    static constexpr int OFF_BAR = OFF_V + NV * TILE;
    // barriers: k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], v_loaded[NV], s_full[NSBUF],
    //           p_ready[NSBUF], o_done[NSBUF], o_final, q_ready, drain, q_loaded, drain_pv
    static constexpr int NBAR = 2 * NK + 3 * NV + 3 * NSBUF + 5;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;     // tmem base, abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM = (SMEM_USED + 1024 > kPfMinSmem ? SMEM_USED + 1024 : kPfMinSmem);
    static_assert(SMEM <= 227 * 1024, "prefill shared memory budget");
    static_assert(kColS + NSBUF * S_BUF <= (int)kPfTmemCols && kColO + PV_SPLIT * D <= kColS && D <= 128,
                  "TMEM budget");
};

struct PfBars {
    uint32_t k_full, k_empty, v_full, v_empty, v_loaded, s_full, p_ready, o_done, o_final, q_ready, drain, q_loaded,
        drain_pv;
};

template <int NK, int NV, int NSB>
__device__ __forceinline__ PfBars pf_bars(uint32_t base) {
    PfBars b;
    b.k_full = base;
    b.k_empty = b.k_full + 8 * NK;
    b.v_full = b.k_empty + 8 * NK;
    b.v_empty = b.v_full + 8 * NV;
    b.v_loaded = b.v_empty + 8 * NV;
    b.s_full = b.v_loaded + 8 * NV;
    b.p_ready = b.s_full + 8 * NSB;
    b.o_done = b.p_ready + 8 * NSB;
    b.o_final = b.o_done + 8 * NSB;
    b.q_ready = b.o_final + 8;
    b.drain = b.q_ready + 8;
    b.q_loaded = b.drain + 8;
    b.drain_pv = b.q_loaded + 8;
    return b;
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, float* __restrict__ o, int B, int S, int H, int Hk,
                  int causal, const int* __restrict__ seq_lens, float scale_log2, int n_qtiles,
                  unsigned int* __restrict__ flags) {
    using C = PfCfg<D>;
    constexpr int BN = C::BN;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    const PfBars bar = pf_bars<C::NK, C::NV, C::NSBUF>(smem_addr(smem + C::OFF_BAR));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = B * H;
    const int tile = n_qtiles - 1 - (int)(blockIdx.x / BH);   // heaviest causal tiles first
    const int bh = (int)(blockIdx.x % BH);
    const int b = bh / H, h = bh % H, g = h / (H / Hk);
    const int q0 = tile * kPfBM;

    int len = S;
    if (seq_lens) {
        len = __ldg(seq_lens + b);
        if (len > S) { len = S; if (threadIdx.x == 0 && tile == n_qtiles - 1) atomicOr(flags, RKV_FLAG_LEN_CLAMPED); }
        if (len < 0) { len = 0; if (threadIdx.x == 0 && tile == n_qtiles - 1) atomicOr(flags, RKV_FLAG_NEGATIVE_INPUT); }
    }
    // keys this tile needs: [0, kv_end)
    const int kv_end = q0 >= len ? 0 : (causal ? min(len, q0 + kPfBM) : len);
    const int nblk = (kv_end + BN - 1) / BN;
    const int64_t q_row = (int64_t)H * D;

    // ------------------------------------------------------------------ setup
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kPfTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NK; ++s) {
            mbar_init(bar.k_full + 8 * s, 1);
            mbar_init(bar.k_empty + 8 * s, 1);
        }
        for (int s = 0; s < C::NV; ++s) {
            mbar_init(bar.v_full + 8 * s, 128);
            mbar_init(bar.v_empty + 8 * s, 1);
            mbar_init(bar.v_loaded + 8 * s, 1);
        }
        for (int s = 0; s < C::NSBUF; ++s) {
            mbar_init(bar.s_full + 8 * s, 1);
            mbar_init(bar.p_ready + 8 * s, 128);
            mbar_init(bar.o_done + 8 * s, 1);
        }
        mbar_init(bar.o_final, 1);
        mbar_init(bar.q_ready, 128);
        mbar_init(bar.drain, 1);
        mbar_init(bar.q_loaded, 1);
        mbar_init(bar.drain_pv, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (nblk > 0) {
        if (warp == 0) {
            // ============================================================ K and V producers
            // lane 0 streams K tiles, lane 16 streams V tiles (both by TMA, same box shape)
            if (lane == 0 || lane == 16) {
                const bool is_k = lane == 0;
                const int NS = is_k ? C::NK : C::NV;
                const uint32_t empty0 = is_k ? bar.k_empty : bar.v_empty;
                const uint32_t full0 = is_k ? bar.k_full : bar.v_loaded;
                const int off0 = is_k ? C::OFF_K : C::OFF_V;
                const void* tm = is_k ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
                bool q_issued = false;
                if (is_k) {       // the query tile, staged in V slots 1 .. QSLOTS
                    mbar_arrive_expect_tx(bar.q_loaded, kPfBM * D * 4);
                    const uint32_t qdst = smem_addr(smem + C::OFF_V + C::TILE);
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d(qdst + c * kPfBM * C::CH * 4, &tm_q, h * D + c * C::CH, q0, b, bar.q_loaded);
                    q_issued = true;
                }
                int issued = 0;
                for (int j = 0; j < nblk; ++j) {
                    const int s = j % NS;
                    const uint32_t ph = (uint32_t)(j / NS) & 1u;
                    if (!is_k && j == 1 && !mbar_wait(bar.q_ready, 0, abort_flag, flags)) break;   // Q consumed
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, flags)) break;
                    const uint32_t full = full0 + 8 * s;
                    mbar_arrive_expect_tx(full, C::TILE);
                    const uint32_t dst = smem_addr(smem + off0);
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d(dst + (is_k ? C::koff(s, c) : s * C::TILE + c * BN * C::CH * 4), tm,
                                    g * D + c * C::CH, j * BN, b, full);
                    issued = j + 1;
                }
                if (*abort_flag) {   // unwinding: let issued copies land
                    for (int j = max(0, issued - NS); j < issued; ++j)
                        mbar_drain(full0 + 8 * (j % NS), (uint32_t)(j / NS) & 1u, 100000000ull);
                    if (q_issued) mbar_drain(bar.q_loaded, 0, 100000000ull);
                }
            }
        } else if (warp == 1 || warp == kPfPvWarp) {
            // ============================================================ MMA issuers
            // Two threads issue: warp 1 the QK^T MMAs, warp 10 the PV MMAs.  A thread needs
            // ~45 cycles per tcgen05.mma it issues, more than one N=64 MMA takes to run,
            // so a single issuer would starve the tensor core.
            if (lane == 0) {
                const bool qk_role = warp == 1;
                constexpr uint32_t id_qk = idesc_tf32(kPfBM, BN, false);
                constexpr uint32_t id_pv = idesc_tf32(kPfBM, D, false);
                bool ok = true;
                int issued_any = 0;
                // Descriptors are built once per ring stage; a k step only adds its byte
                // offset (>> 4) to the start-address field, which cannot carry out of it
                // (shared addresses are below 2^18).
                const uint64_t kdesc0 = smem_desc(smem_addr(smem + C::OFF_K), 16, C::K_ATOM, C::K_SWIZZLE);
                const uint64_t vdesc0 = smem_desc(smem_addr(smem + C::OFF_V), 16, 1024, kSwizzle128B);
                if (qk_role) {
                    ok = mbar_wait(bar.q_ready, 0, abort_flag, flags);
                    // S_j goes to buffer j % NSBUF (paired blocks: two adjacent buffers); before
                    // QK_j overwrites the buffer of block j - NSBUF, PV_{j-NSBUF} must have
                    // finished reading P from it.  The wait is exact: PV_{j-2*NSBUF} completed
                    // before QK_{j-NSBUF} was issued, and PV_j cannot have started (it needs S_j).
                    constexpr uint32_t id_qk2 = idesc_tf32(kPfBM, 2 * BN, false);
                    for (int j = 0; ok && j < nblk; j += C::KPAIR ? 2 : 1) {
                        const int nb = (C::KPAIR && j + 1 < nblk) ? 2 : 1;   // blocks in this chain
                        for (int bb = j; ok && bb < j + nb; ++bb) {
                            if (bb >= C::NSBUF)
                                ok = mbar_wait(bar.o_done + 8 * (bb % C::NSBUF),
                                               (uint32_t)((bb - C::NSBUF) / C::NSBUF) & 1u, abort_flag, flags);
                            if (ok)
                                ok = mbar_wait(bar.k_full + 8 * (bb % C::NK), (uint32_t)(bb / C::NK) & 1u, abort_flag,
                                               flags);
                        }
                        if (!ok) break;
                        tc_fence_after();
                        const int s = j % C::NK;          // even when paired: slots s, s+1 share a pair
                        const uint32_t d_tmem = tmem + kColS + (uint32_t)((j % C::NSBUF) * C::S_BUF);
#pragma unroll
                        for (int k = 0; k < D / 8; ++k) {
                            const int c = k / (C::CH / 8), kk = k % (C::CH / 8);
                            const uint64_t bdesc = kdesc0 + (uint64_t)((C::koff(s, c) + kk * 32) >> 4);
                            mma_tf32_ts(d_tmem, tmem + kColQ + 8 * k, bdesc, nb == 2 ? id_qk2 : id_qk, k > 0 ? 1u : 0u);
                        }
                        for (int bb = j; bb < j + nb; ++bb) {
                            mma_commit(bar.s_full + 8 * (bb % C::NSBUF));
                            mma_commit(bar.k_empty + 8 * (bb % C::NK));
                        }
                        issued_any = 1;
                    }
                    if (!ok && issued_any) {   // unwinding: let issued MMAs finish before TMEM is freed
                        mma_commit(bar.drain);
                        mbar_drain(bar.drain, 0, 100000000ull);
                    }
                } else {
                    for (int pj = 0; ok && pj < nblk; ++pj) {
                        // O += P_pj V_pj
                        const int sv = pj % C::NV, sb = pj % C::NSBUF;
                        if (!(ok = mbar_wait(bar.p_ready + 8 * sb, (uint32_t)(pj / C::NSBUF) & 1u, abort_flag, flags))) break;
                        if (!(ok = mbar_wait(bar.v_full + 8 * sv, (uint32_t)(pj / C::NV) & 1u, abort_flag, flags))) break;
                        tc_fence_after();
                        const uint64_t vd = vdesc0 + (uint64_t)(sv * (C::TILE >> 4));
                        const uint32_t a_tmem = tmem + kColS + (uint32_t)(sb * C::S_BUF);
                        const uint32_t first = pj > 0 ? 1u : 0u;
#pragma unroll
                        for (int k = 0; k < BN / 8; ++k) {
                            // V^T tile: rows = d, 32 keys per 128-byte row, key chunks D*128 bytes apart
                            const uint64_t bdesc = vd + (uint64_t)(((k / 4) * (D * 128) + (k % 4) * 32) >> 4);
                            const int part = k % C::PV_SPLIT;
                            mma_tf32_ts(tmem + kColO + part * D, a_tmem + 8 * k, bdesc, id_pv,
                                        k >= C::PV_SPLIT ? 1u : first);
                        }
                        mma_commit(bar.o_done + 8 * sb);
                        mma_commit(bar.v_empty + 8 * sv);
                        issued_any = 1;
                    }
                    if (ok) {
                        mma_commit(bar.o_final);
                    } else if (issued_any) {
                        mma_commit(bar.drain_pv);
                        mbar_drain(bar.drain_pv, 0, 100000000ull);
                    }
                }
            }
        } else if (warp >= kPfVWarp0 && warp < kPfVWarp0 + 4) {
            // ============================================================ V transposer
            // V tiles arrive by TMA in the same swizzled layout as K (rows = keys).  The
            // transposer rewrites each slot in place as V^T: work item = (key quad aa,
            // d quad dq), a 4x4 block read with four 16-byte loads and written as four
            // 16-byte rows of V^T.  Lane numbering puts 4 consecutive key quads x 2 d
            // quads (D = 16: 8 key quads x 1) in each quarter-warp, so its eight V^T
            // stores hit eight distinct 128-byte-swizzle chunks: no conflicts.
            const int wv = warp - kPfVWarp0;                      // 0..3
            constexpr int LDQ = D / 4 < 8 ? D / 4 : 8;           // lanes along d quads
            constexpr int LAA = 32 / LDQ;                        // lanes along key quads
            constexpr int GA = (BN / 4) / LAA;                   // lane groups along keys
            constexpr int GD = (D / 4) / LDQ;                    // lane groups along d
            constexpr int PER = GA * GD / 4;                     // groups per warp
            static_assert(GA * GD % 4 == 0 && PER >= 1, "V transposer work split");
            const int aa_lo = lane % LAA, dq_lo = lane / LAA;
            // Byte offset of V[key][d] in a TMA-staged tile (box {CH floats, BN keys} per
            // d chunk, swizzled: 16-byte chunk index XOR key bits).
            auto staged = [](int key, int dq) -> int {
                if constexpr (D >= 32)
                    return (dq >> 3) * (BN * 128) + key * 128 + (((dq & 7) ^ (key & 7)) << 4);
                else
                    return key * 64 + (((dq & 3) ^ ((key >> 1) & 3)) << 4);
            };
            for (int j = 0; j < nblk; ++j) {
                const int s = j % C::NV;
                unsigned char* vt = smem + C::OFF_V + s * C::TILE;
                if (!mbar_wait(bar.v_loaded + 8 * s, (uint32_t)(j / C::NV) & 1u, abort_flag, flags)) break;
                float4 x[PER][4];
#pragma unroll
                for (int it = 0; it < PER; ++it) {
                    const int G = it * 4 + wv;
                    const int aa = (G % GA) * LAA + aa_lo;
                    const int dq = (G / GA) * LDQ + dq_lo;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int key = aa * 4 + r;
                        // keys past the sequence end were zero-filled by the copy engine
                        x[it][r] = *reinterpret_cast<const float4*>(vt + staged(key, dq));
                    }
                }
                named_barrier(2, 128);        // every thread has read its blocks: rewrite in place
#pragma unroll
                for (int it = 0; it < PER; ++it) {
                    const int G = it * 4 + wv;
                    const int aa = (G % GA) * LAA + aa_lo;
                    const int dq = (G / GA) * LDQ + dq_lo;
                    const int kc = aa >> 3;                      // 32-key chunk of the V^T row
                    const float4 c0 = x[it][0], c1 = x[it][1], c2 = x[it][2], c3 = x[it][3];
                    const uint4 w[4] = {
                        make_uint4(round_tf32(c0.x), round_tf32(c1.x), round_tf32(c2.x), round_tf32(c3.x)),
                        make_uint4(round_tf32(c0.y), round_tf32(c1.y), round_tf32(c2.y), round_tf32(c3.y)),
                        make_uint4(round_tf32(c0.z), round_tf32(c1.z), round_tf32(c2.z), round_tf32(c3.z)),
                        make_uint4(round_tf32(c0.w), round_tf32(c1.w), round_tf32(c2.w), round_tf32(c3.w))};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int d = dq * 4 + i;
                        const int off = kc * (D * 128) + d * 128 + (((aa & 7) ^ (d & 7)) << 4);
                        *reinterpret_cast<uint4*>(vt + off) = w[i];
                    }
                }
                fence_proxy_async();          // generic-proxy stores -> tensor-core reads
                mbar_arrive(bar.v_full + 8 * s);
            }
        } else {
            // ============================================================ softmax / epilogue
            const int quad = warp & 3;                       // TMEM lane quadrant of this warp
            const int r = quad * 32 + lane;                  // query row within the tile
            const int qi = q0 + r;
            const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
            // Q row -> TMEM (pre-scaled, rounded to TF32), read from the TMA-staged tile
            {
                bool qok = mbar_wait(bar.q_loaded, 0, abort_flag, flags);
                qok = __all_sync(0xffffffffu, qok);
                const unsigned char* qs = smem + C::OFF_V + C::TILE;
                auto qv = [&](int dq) -> float4 {     // Q[r][4dq .. 4dq+3] in the swizzled staging
                    if constexpr (D >= 32)
                        return *reinterpret_cast<const float4*>(qs + (dq >> 3) * (kPfBM * 128) + r * 128 +
                                                                (((dq & 7) ^ (r & 7)) << 4));
                    else
                        return *reinterpret_cast<const float4*>(qs + r * 64 + (((dq & 3) ^ ((r >> 1) & 3)) << 4));
                };
                if (qok) {
                    if constexpr (D >= 32) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t w[32];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float4 t4 = qv(c * 8 + e);
                                w[4 * e + 0] = round_tf32(t4.x * scale_log2);
                                w[4 * e + 1] = round_tf32(t4.y * scale_log2);
                                w[4 * e + 2] = round_tf32(t4.z * scale_log2);
                                w[4 * e + 3] = round_tf32(t4.w * scale_log2);
                            }
                            tmem_st32(lane_base + kColQ + 32 * c, w);
                        }
                    } else {
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 t4 = qv(e);
                            w[4 * e + 0] = round_tf32(t4.x * scale_log2);
                            w[4 * e + 1] = round_tf32(t4.y * scale_log2);
                            w[4 * e + 2] = round_tf32(t4.z * scale_log2);
                            w[4 * e + 3] = round_tf32(t4.w * scale_log2);
                        }
                        tmem_st16(lane_base + kColQ, w);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(bar.q_ready);
            }
            float m_run = -INFINITY, l_run = 0.0f;
            bool ok = true;
            const int key_lim = causal ? min(qi + 1, len) : len;   // keys visible to this row
            for (int j = 0; j < nblk; ++j) {
                ok = mbar_wait(bar.s_full + 8 * (j % C::NSBUF), (uint32_t)(j / C::NSBUF) & 1u, abort_flag, flags);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;   // warp-uniform before TMEM access
                tc_fence_after();
                const uint32_t s_col = lane_base + kColS + (uint32_t)((j % C::NSBUF) * C::S_BUF);
                float s[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t w[32];
                    tmem_ld32(s_col + 32 * c, w);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[32 * c + e] = __uint_as_float(w[e]);
                }
                const int k0 = j * BN;
                const int nvis = min(max(key_lim - k0, 0), BN);     // visible keys of this block
                if (__any_sync(0xffffffffu, nvis < BN)) {
#pragma unroll
                    for (int e = 0; e < BN; ++e)
                        if (e >= nvis) s[e] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) mx[t] = s[t];
#pragma unroll
                for (int e = 8; e < BN; ++e) mx[e & 7] = fmaxf(mx[e & 7], s[e]);
                const float m_blk = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                          fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                const bool need = m_blk > m_run + kLazyRescale;
                const float m_use = need ? m_blk : m_run;
                const float alpha = need ? fast_exp2(m_run - m_blk) : 1.0f;
                // p = 2^(s - m); the tensor core truncates f32 operands to TF32, so p is
                // truncated here too and the row sum is taken over exactly those values
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t w[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float x = s[32 * c + e];
                        const float p = (x == -INFINITY) ? 0.0f : fast_exp2(x - m_use);
                        w[e] = __float_as_uint(p) & 0xFFFFE000u;
                        ls[e & 7] += __uint_as_float(w[e]);
                    }
                    tmem_st32(s_col + 32 * c, w);
                }
                const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                l_run = l_run * alpha + lsum;
                m_run = m_use;
                tmem_wait_st();
                if (j > 0 && __any_sync(0xffffffffu, need)) {
                    // O holds blocks < j once PV_{j-1} completes; scale it by alpha.  Seeing S_j
                    // means PV_{j-NSBUF} completed (issued before QK_j), so the barrier of
                    // PV_{j-1}'s buffer is at most one phase behind: the parity wait is exact.
                    ok = mbar_wait(bar.o_done + 8 * ((j - 1) % C::NSBUF), (uint32_t)((j - 1) / C::NSBUF) & 1u,
                                   abort_flag, flags);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < C::PV_SPLIT * ((D + 31) / 32); ++c) {
                        if constexpr (D >= 32) {
                            uint32_t w[32];
                            tmem_ld32(lane_base + kColO + 32 * c, w);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
                            tmem_st32(lane_base + kColO + 32 * c, w);
                        } else {
                            uint32_t w[16];
                            tmem_ld16(lane_base + kColO + 16 * c, w);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
                            tmem_st16(lane_base + kColO + 16 * c, w);
                        }
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(bar.p_ready + 8 * (j % C::NSBUF));
            }
            // ---------------------------------------------------------- epilogue
            if (ok) ok = mbar_wait(bar.o_final, 0, abort_flag, flags);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                const float inv = (qi < len && l_run > 0.0f) ? 1.0f / l_run : 0.0f;
                float4* op = reinterpret_cast<float4*>(o + ((int64_t)b * S + qi) * q_row + (int64_t)h * D);
#pragma unroll
                for (int c = 0; c < (D + 31) / 32; ++c) {
                    if constexpr (D >= 32) {
                        uint32_t w[32];
                        tmem_ld32(lane_base + kColO + 32 * c, w);
                        if constexpr (C::PV_SPLIT == 2) {
                            uint32_t w2[32];
                            tmem_ld32(lane_base + kColO + D + 32 * c, w2);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) + __uint_as_float(w2[e]));
                        } else {
                            tmem_wait_ld();
                        }
                        if (qi < S) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                __stcs(op + c * 8 + e,     // streaming: written once, not re-read here
                                       make_float4(__uint_as_float(w[4 * e]) * inv, __uint_as_float(w[4 * e + 1]) * inv,
                                                   __uint_as_float(w[4 * e + 2]) * inv, __uint_as_float(w[4 * e + 3]) * inv));
                        }
                    } else {
                        uint32_t w[16], w2[16];
                        tmem_ld16(lane_base + kColO, w);
                        tmem_ld16(lane_base + kColO + D, w2);     // D = 16 always splits PV
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) + __uint_as_float(w2[e]));
                        if (qi < S) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                __stcs(op + e, make_float4(__uint_as_float(w[4 * e]) * inv, __uint_as_float(w[4 * e + 1]) * inv,
                                                           __uint_as_float(w[4 * e + 2]) * inv, __uint_as_float(w[4 * e + 3]) * inv));
                        }
                    }
                }
            }
        }
    } else if (warp >= kPfSoftmaxWarp0 && warp < kPfVWarp0) {
        // no key is visible to any row of this tile: the rows are padding -> zeros
        const int r = (warp & 3) * 32 + lane;
        const int qi = q0 + r;
        if (qi < S) {
            float4* op = reinterpret_cast<float4*>(o + ((int64_t)b * S + qi) * q_row + (int64_t)h * D);
#pragma unroll
            for (int e = 0; e < D / 4; ++e) op[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kPfTmemCols);
    }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <int D>
static rkv_status launch_prefill_tc_t(const PrefillArgs& a, cudaStream_t stream) {
    using C = PfCfg<D>;
    auto encode = tensor_map_encoder();
    if (!encode) return set_error(RKV_ERR_LAUNCH, "attn_prefill: cuTensorMapEncodeTiled unavailable");
    CUtensorMap tm_k, tm_v, tm_q;
    const cuuint64_t dims[3] = {(cuuint64_t)a.Hk * D, (cuuint64_t)a.S, (cuuint64_t)a.B};
    const cuuint64_t strides[2] = {(cuuint64_t)a.Hk * D * 4, (cuuint64_t)a.S * a.Hk * D * 4};
    const cuuint32_t box[3] = {(cuuint32_t)C::CH, (cuuint32_t)C::BN, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw = D >= 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult cr = encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.k), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr == CUDA_SUCCESS)
        cr = encode(&tm_v, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.v), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr == CUDA_SUCCESS) {
        const cuuint64_t qdims[3] = {(cuuint64_t)a.H * D, (cuuint64_t)a.S, (cuuint64_t)a.B};
        const cuuint64_t qstrides[2] = {(cuuint64_t)a.H * D * 4, (cuuint64_t)a.S * a.H * D * 4};
        const cuuint32_t qbox[3] = {(cuuint32_t)C::CH, (cuuint32_t)kPfBM, 1};
        cr = encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.q), qdims, qstrides, qbox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS) return set_error(RKV_ERR_LAUNCH, "attn_prefill: tensor map encode failed (%d)", (int)cr);
    auto kern = prefill_tc_kernel<D>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return check_launch("attn_prefill: shared-memory attribute");
        attr_done[dev] = true;
    }
    const int n_qtiles = (a.S + kPfBM - 1) / kPfBM;
    const int64_t grid = (int64_t)n_qtiles * a.B * a.H;
    if (grid > 0x7FFFFFFF) return set_error(RKV_ERR_UNSUPPORTED, "attn_prefill: grid too large");
    kern<<<(unsigned)grid, kPfThreads, C::SMEM, stream>>>(tm_k, tm_v, tm_q, a.o, a.B, a.S, a.H, a.Hk, a.causal ? 1 : 0,
                                                           a.seq_lens, a.scale * kPfLog2e, n_qtiles, a.flags);
    return check_launch("attn_prefill");
}

rkv_status launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    switch (a.D) {
        case 16: return launch_prefill_tc_t<16>(a, stream);
        case 32: return launch_prefill_tc_t<32>(a, stream);
        case 64: return launch_prefill_tc_t<64>(a, stream);
        case 128: return launch_prefill_tc_t<128>(a, stream);
    }
    return set_error(RKV_ERR_UNSUPPORTED, "attn_prefill: head_dim %d", a.D);
}

}  // namespace rkv
