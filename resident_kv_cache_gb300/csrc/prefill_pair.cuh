#pragma once
// prefill_pair.cuh -- the grouped-query prefill on a CTA pair (sm_103a, head_dim 128).
//
// Semantics: the same as prefill_tc.cuh (trueno-gpu 0.4.11 src/memory/resident/attention.rs,
// fn batched_multihead_attention_optimized; trustformers-core 0.2.0
// src/gpu_ops/cuda/oxicuda/attention.rs, fn attention_prefill_gpu_to_gpu): per (batch, head),
// softmax(Q K^T * scale) V over the keys each query sees, causal or not.
//
// With grouped-query attention two query heads of one kv group read the same keys and values.
// Here the two CTAs of a cluster take such a pair of heads over the same 128-query tile and share
// every tensor-core product: one tcgen05.mma of M = 256 (cta_group::2), issued by the even CTA,
// holds head 2i's 128 query rows in the even CTA and head 2i+1's in the odd one.  B, the key
// block (QK^T) or the transposed value block (PV), is split by its N rows across the two CTAs:
//   S_j (256 x 128 keys) = Q (256 x 128, each CTA's rows in its own shared memory)
//                          . K_j^T (each CTA holds 64 of the block's 128 keys)
//   O   (256 x 128 d)   += P_j (each CTA's 128 rows in its own TMEM) . V_j (each CTA holds V^T for
//                          64 of the 128 head dimensions)
// Both heads see the same keys under the same mask, so no product is wasted.  Compared with one
// CTA per head, each CTA loads, holds and transposes half of every K and V block, one warp
// issues the products of both, and the query tile sits in shared memory rather than in tensor
// memory, which leaves room for three 128-key score buffers (384 keys in flight against 256).
//
// Roles (12 warps, as in prefill_tc.cuh), in each CTA of the pair:
//   warp 0       K producer: per item this CTA's query rows (its head) into the Q buffer, once
//                the previous item's QK^T is done with it; then per block this CTA's 64 keys by
//                TMA, completing on the even CTA's k_full barrier.
//   warp 11      V producer: per block this CTA's 64 head dimensions of 128 value rows by TMA;
//                per item two output staging fills and the TMA stores of O.
//   warp 1, 10   (even CTA only) QK^T and PV issuers (whole warps, one elected lane issuing);
//                warp 1 also allocates tensor memory.
//   warps 2-5    softmax / epilogue, one thread per query row (TMEM lane), as in prefill_tc.cuh.
//   warps 6-9    round the query tile to nearest TF32 in place; transpose each V block in place.
// Barriers the issuers wait on live in the even CTA and count one arrival per warp from both
// CTAs (8); barriers the issuers signal get one multicast commit into both CTAs.
#include "prefill_tc.cuh"

namespace rkv {

struct PpCfg {
    static constexpr int D = 128;                       // head_dim
    static constexpr int BN = 128;                      // keys per block
    static constexpr int CH = 32;                       // floats per 128-byte swizzled row chunk
    static constexpr int NCH = D / CH;
    static constexpr int NK = 2, NV = 3, NSBUF = 3;     // K stages, V stages, S/P buffers
    static constexpr int OSLOTS = 2, OCH = 2;           // output staging: 2 V slots x 2 column chunks
    static constexpr int QT = kPfBM * D * 4;            // query tile: 4 chunks x 128 rows x 128 B
    static constexpr int QCH = kPfBM * CH * 4;          //   one chunk (16 KB)
    static constexpr int KT = (BN / 2) * D * 4;         // this CTA's K half: 4 chunks x 64 keys x 128 B
    static constexpr int KCH = (BN / 2) * CH * 4;       //   one chunk (8 KB)
    static constexpr int VT = BN * (D / 2) * 4;         // this CTA's V half (32 KB): as loaded, 2 d chunks
    static constexpr int VCH = BN * CH * 4;             //   x 128 keys x 128 B; as V^T, 4 key chunks x
    static constexpr int VTCH = (D / 2) * CH * 4;       //   64 d rows x 128 B (8 KB each)
    static constexpr int OFF_Q = 0, OFF_K = QT, OFF_V = OFF_K + NK * KT, OFF_BAR = OFF_V + NV * VT;
    enum : int {
        B_KFULL = 0,                    // [NK]  even CTA: 1 arrival + both halves' bytes
        B_KEMPTY = B_KFULL + NK,        // [NK]  multicast commit
        B_VLOADED = B_KEMPTY + NK,      // [NV]  local: this CTA's V half landed / staging slot handed out
        B_VFULL = B_VLOADED + NV,       // [NV]  even CTA: V^T written, 4 warps x 2 CTAs
        B_VEMPTY = B_VFULL + NV,        // [NV]  multicast commit, or the local store of a staging slot
        B_SFULL = B_VEMPTY + NV,        // [NSBUF] multicast commit
        B_PREADY = B_SFULL + NSBUF,     // [NSBUF] even CTA: P written, 4 warps x 2 CTAs
        B_ODONE = B_PREADY + NSBUF,     // [NSBUF] multicast commit
        B_OFINAL = B_ODONE + NSBUF,     // multicast commit: the item's last PV done
        B_OFREE,                        // even CTA: O read out, 4 warps x 2 CTAs
        B_OSTAGED,                      // [OSLOTS] local: the epilogue's 128 threads staged O
        B_QFREE = B_OSTAGED + OSLOTS,   // multicast commit: the item's last QK^T done
        B_QLOADED,                      // local: the query tile landed
        B_QREADY,                       // even CTA: query tile rounded, 4 warps x 2 CTAs
        B_FIN,                          // multicast commits from both issuers at the end
        NBAR
    };
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // tmem base, abort flag
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static_assert(SMEM <= 227 * 1024, "pair prefill shared memory budget");
    static constexpr uint32_t COL_O = 0, COL_S = D;       // TMEM columns: O, then NSBUF S buffers
    static_assert(COL_S + NSBUF * BN <= kPfTmemCols, "pair prefill TMEM budget");
};

// One work item: a 128-query tile of the head pair (2 hp, 2 hp + 1) of kv group g in batch b;
// h is this CTA's head.  Query i sits at key position p0 + i; the sequence has n_kv keys.
struct PpWork {
    int b, g, h, q0, len, p0, n_kv, nblk;
};

// Items are numbered heaviest causal tiles first, like pf_work.
__device__ __forceinline__ PpWork pp_work(int u, uint32_t rank, int B, int H, int Hk, int S, int n_qtiles, int causal,
                                          const int* __restrict__ seq_lens, const PfKv& kv) {
    const int G = H / Hk, HP = G / 2;
    const int per_tile = B * Hk * HP;
    PpWork w;
    const int tile = n_qtiles - 1 - u / per_tile;
    const int rem = u % per_tile;
    w.b = rem / (Hk * HP);
    const int x = rem % (Hk * HP);
    w.g = x / HP;
    w.h = w.g * G + 2 * (x % HP) + (int)rank;
    w.q0 = tile * kPfBM;
    w.len = seq_lens ? min(max(__ldg(seq_lens + w.b), 0), S) : S;
    w.p0 = kv.start ? min(max(__ldg(kv.start + w.b), 0), kv.cap) : 0;
    w.n_kv = min(w.p0 + w.len, kv.cap);
    const int kv_end = w.q0 >= w.len ? 0 : (causal ? min(w.n_kv, w.p0 + w.q0 + kPfBM) : w.n_kv);
    w.nblk = (kv_end + PpCfg::BN - 1) / PpCfg::BN;
    return w;
}

// The k-th item of this CTA's cluster: dealt like pf_item, over clusters.
__device__ __forceinline__ int pp_item(int k) {
    const int NC = (int)gridDim.x >> 1, ci = (int)blockIdx.x >> 1;
    return k * NC + ((k & 1) ? NC - 1 - ci : ci);
}

// GUARD and FILL as in prefill_tc.cuh: tiles that may reach past a sequence, and a launch
// followed by the programmatic-dependent cache fill, which this kernel releases at once; the
// FILL variant is held to kPfFillRegs registers a thread so that the fill's blocks fit beside it.
template <bool GUARD, bool FILL>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(FILL ? kPfFillRegs : 65536 / kPfThreads / 8 * 8)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                    float* __restrict__ o, int B, int S, int H, int Hk, int causal, const int* __restrict__ seq_lens,
                    float scale_log2, int n_qtiles, int n_work, const PfKv kv, unsigned int* __restrict__ flags) {
    using C = PpCfg;
    constexpr int D = C::D, BN = C::BN;
    static_assert(!(FILL && GUARD), "the fused cache fill is built for whole sequences only");
    if (FILL) griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    const uint32_t bar0 = smem_addr(smem + C::OFF_BAR);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };                      // this CTA's barrier i
    auto LEAD = [&](int i) { return cluster_map(bar0 + 8u * (uint32_t)i, 0); };     // the even CTA's
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const uint32_t rank = cluster_rank();
    const uint32_t peer_abort = cluster_map(smem_addr(smem + C::OFF_MISC + 4), rank ^ 1u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t q_row = (int64_t)H * D;
    auto work = [&](int u) { return pp_work(u, rank, B, H, Hk, S, n_qtiles, causal, seq_lens, kv); };

    if ((seq_lens || kv.start) && blockIdx.x == 0) {     // report clamped lengths once per launch
        for (int i = threadIdx.x; i < B; i += blockDim.x) {
            const int l = seq_lens ? __ldg(seq_lens + i) : S;
            const int p = kv.start ? __ldg(kv.start + i) : 0;
            if (l > S || (int64_t)max(p, 0) + min(max(l, 0), S) > kv.cap) atomicOr(flags, RKV_FLAG_LEN_CLAMPED);
            if (l < 0 || p < 0) atomicOr(flags, RKV_FLAG_NEGATIVE_INPUT);
        }
    }

    // ------------------------------------------------------------------ setup
    if (warp == 1) {                  // one warp of each CTA allocates for the pair together
        tmem_alloc_pair(smem_addr(tmem_slot), kPfTmemCols);
        tmem_relinquish_pair();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NK; ++s) {
            mbar_init(BAR(C::B_KFULL + s), 1);
            mbar_init(BAR(C::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < C::NV; ++s) {
            mbar_init(BAR(C::B_VLOADED + s), 1);
            mbar_init(BAR(C::B_VFULL + s), 8);
            mbar_init(BAR(C::B_VEMPTY + s), 1);
        }
        for (int s = 0; s < C::NSBUF; ++s) {
            mbar_init(BAR(C::B_SFULL + s), 1);
            mbar_init(BAR(C::B_PREADY + s), 8);
            mbar_init(BAR(C::B_ODONE + s), 1);
        }
        mbar_init(BAR(C::B_OFINAL), 1);
        mbar_init(BAR(C::B_OFREE), 8);
        for (int i = 0; i < C::OSLOTS; ++i) mbar_init(BAR(C::B_OSTAGED + i), 128);
        mbar_init(BAR(C::B_QFREE), 1);
        mbar_init(BAR(C::B_QLOADED), 1);
        mbar_init(BAR(C::B_QREADY), 8);
        mbar_init(BAR(C::B_FIN), 2);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_o);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                   // both CTAs' barriers exist before anything crosses over
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Every role walks the same item sequence (the same in both CTAs) and numbers key blocks and
    // ring fills with running counters across items, as in prefill_tc.cuh.
    if (warp == 0) {
        // ================================================================ K producer
        if (lane == 0) {
            int f = 0, t = 0;         // K-ring fills, items with keys
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int u = pp_item(k);
                if (u >= n_work) break;
                const PpWork w = work(u);
                if (w.nblk == 0) continue;
                {                     // the next item's query rows -> L2, ahead of their own copy
                    const int un = pp_item(k + 1);
                    if (un < n_work) {
                        const PpWork wn = work(un);
#pragma unroll
                        for (int c = 0; c < C::NCH; ++c) tma_prefetch_l2_3d(&tm_q, wn.h * D + c * C::CH, wn.q0, wn.b);
                    }
                }
                // this head's query tile, once the previous item's QK^T products no longer read it
                if (t > 0 && !(ok = mbar_wait(BAR(C::B_QFREE), (uint32_t)(t - 1) & 1u, abort_flag, flags))) break;
                mbar_arrive_expect_tx(BAR(C::B_QLOADED), C::QT);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(smem_addr(smem + C::OFF_Q + c * C::QCH), &tm_q, w.h * D + c * C::CH, w.q0, w.b,
                                BAR(C::B_QLOADED));
                ++t;
                for (int j = 0; j < w.nblk; ++j, ++f) {
                    const int s = f % C::NK;
                    if (!(ok = mbar_wait(BAR(C::B_KEMPTY + s), ((uint32_t)(f / C::NK) & 1u) ^ 1u, abort_flag, flags)))
                        break;
                    if (rank == 0) mbar_arrive_expect_tx(BAR(C::B_KFULL + s), 2 * C::KT);
                    const uint32_t full = LEAD(C::B_KFULL + s);
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d_pair(smem_addr(smem + C::OFF_K + s * C::KT + c * C::KCH), &tm_k,
                                         w.g * kv.xg + c * C::CH, j * BN + (int)rank * (BN / 2),
                                         w.b * kv.zb + w.g * kv.zg, full);
                }
            }
            if (!ok) st_cluster_u32(peer_abort, 1u);
            if (*abort_flag) {        // unwinding: let issued copies land
                if (t > 0) mbar_drain(BAR(C::B_QLOADED), (uint32_t)(t - 1) & 1u, 100000000ull);
                if (rank == 0)
                    for (int g = max(0, f - C::NK); g < f; ++g)
                        mbar_drain(BAR(C::B_KFULL + g % C::NK), (uint32_t)(g / C::NK) & 1u, 100000000ull);
            }
        }
    } else if (warp == kPfVProdWarp) {
        // ================================================================ V producer / O stores
        if (lane == 0) {
            int gs = 0, t = 0;        // V-ring fills, items with keys
            bool ok = true;
            int pend = -1, pt = 0;    // first staging fill not yet stored (-1: none) and its item
            PpWork pw{};
            auto flush = [&]() -> bool {
                for (int i = 0; i < C::OSLOTS; ++i)
                    if (!mbar_wait(BAR(C::B_OSTAGED + i), (uint32_t)pt & 1u, abort_flag, flags)) return false;
                for (int i = 0; i < C::OSLOTS; ++i) {
                    const uint32_t src = smem_addr(smem + C::OFF_V) + ((pend + i) % C::NV) * C::VT;
#pragma unroll
                    for (int cc = 0; cc < C::OCH; ++cc)
                        tma_store_3d(&tm_o, src + cc * C::QCH, pw.h * D + (i * C::OCH + cc) * C::CH, pw.q0, pw.b);
                }
                bulk_commit();
                bulk_wait_read_all();
                for (int i = 0; i < C::OSLOTS; ++i) mbar_arrive(BAR(C::B_VEMPTY + (pend + i) % C::NV));
                pend = -1;
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int u = pp_item(k);
                if (u >= n_work) break;
                const PpWork w = work(u);
                if (w.nblk == 0) continue;
                for (int j = 0; j < w.nblk + C::OSLOTS; ++j) {
                    if (pend >= 0 && gs >= pend + C::NV && !(ok = flush())) break;
                    const int s = gs % C::NV;
                    if (!(ok = mbar_wait(BAR(C::B_VEMPTY + s), ((uint32_t)(gs / C::NV) & 1u) ^ 1u, abort_flag, flags)))
                        break;
                    if (j >= w.nblk) {      // output staging fill: handed to the epilogue
                        if (j == w.nblk) { pend = gs; pw = w; pt = t; }
                        ++gs;
                        mbar_arrive(BAR(C::B_VLOADED + s));
                        continue;
                    }
                    ++gs;
                    mbar_arrive_expect_tx(BAR(C::B_VLOADED + s), C::VT);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d(smem_addr(smem + C::OFF_V + s * C::VT + c * C::VCH), &tm_v,
                                    w.g * kv.xg + (int)rank * (D / 2) + c * C::CH, j * BN, w.b * kv.zb + w.g * kv.zg,
                                    BAR(C::B_VLOADED + s));
                }
                ++t;
            }
            if (ok && pend >= 0) ok = flush();
            bulk_wait_all();                  // output stores complete before the CTA exits
            if (!ok) st_cluster_u32(peer_abort, 1u);
            if (*abort_flag) {
                for (int g = max(0, gs - C::NV); g < gs; ++g)
                    mbar_drain(BAR(C::B_VLOADED + g % C::NV), (uint32_t)(g / C::NV) & 1u, 100000000ull);
            }
        }
    } else if (warp == 1 || warp == kPfPvWarp) {
        // ================================================================ MMA issuers (even CTA)
        // The whole warp walks the loop (every value in it is warp-uniform); one elected lane
        // executes each MMA and commit, and waits are decided by the warp together.
        if (rank == 0) {
            const bool qk_role = warp == 1;
            constexpr uint32_t id_qk = idesc_tf32(2 * kPfBM, BN, false);
            constexpr uint32_t id_pv = idesc_tf32(2 * kPfBM, D, false);
            bool ok = true;
            int g0 = 0, t = 0, f = 0, fv = 0;
            int vcnt[C::NV] = {};              // V fills (not staging fills) seen per V slot
            const uint64_t qdesc0 = smem_desc(smem_addr(smem + C::OFF_Q), 16, 1024, kSwizzle128B);
            const uint64_t kdesc0 = smem_desc(smem_addr(smem + C::OFF_K), 16, 1024, kSwizzle128B);
            const uint64_t vdesc0 = smem_desc(smem_addr(smem + C::OFF_V), 16, 1024, kSwizzle128B);
            for (int k = 0; ok; ++k) {
                const int u = pp_item(k);
                if (u >= n_work) break;
                const PpWork w = work(u);
                if (w.nblk == 0) continue;
                if (qk_role) {
                    // S of block gb goes to buffer gb % NSBUF once the PV that read P from it
                    // (block gb - NSBUF) has finished; the parity wait is exact as in prefill_tc.cuh.
                    ok = mbar_wait<true>(BAR(C::B_QREADY), (uint32_t)t & 1u, abort_flag, flags);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
                    for (int j = 0; j < w.nblk; ++j, ++f) {
                        const int gb = g0 + j, s = f % C::NK, sb = gb % C::NSBUF;
                        if (gb >= C::NSBUF)
                            ok = mbar_wait(BAR(C::B_ODONE + sb), (uint32_t)((gb - C::NSBUF) / C::NSBUF) & 1u, abort_flag,
                                           flags);
                        if (ok) ok = mbar_wait(BAR(C::B_KFULL + s), (uint32_t)(f / C::NK) & 1u, abort_flag, flags);
                        if (!(ok = __all_sync(0xffffffffu, ok))) break;
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + C::COL_S + (uint32_t)(sb * BN);
#pragma unroll
                        for (int kk8 = 0; kk8 < D / 8; ++kk8) {
                            const int c = kk8 / 4, kk = kk8 % 4;
                            const uint64_t a = qdesc0 + (uint64_t)((c * C::QCH + kk * 32) >> 4);
                            const uint64_t b = kdesc0 + (uint64_t)((s * C::KT + c * C::KCH + kk * 32) >> 4);
                            mma_tf32_ss_pair(d_tmem, a, b, id_qk, kk8 > 0 ? 1u : 0u);
                        }
                        mma_commit_pair(BAR(C::B_SFULL + sb));
                        mma_commit_pair(BAR(C::B_KEMPTY + s));
                    }
                    if (!ok) break;
                    mma_commit_pair(BAR(C::B_QFREE));    // the query tile may be replaced
                } else {
                    // O is reused item after item: a new item's first PV overwrites it only after
                    // both epilogues have read the previous item's O.
                    if (t > 0) ok = mbar_wait<true>(BAR(C::B_OFREE), (uint32_t)(t - 1) & 1u, abort_flag, flags);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    for (int j = 0; j < w.nblk; ++j) {
                        const int gb = g0 + j, sv = (fv + j) % C::NV, sb = gb % C::NSBUF;
                        ok = mbar_wait<true>(BAR(C::B_PREADY + sb), (uint32_t)(gb / C::NSBUF) & 1u, abort_flag, flags);
                        if (!(ok = __all_sync(0xffffffffu, ok))) break;
                        // v_full of a slot completes once per V fill of that slot (staging fills do
                        // not arrive on it), so its phase is counted per slot
                        const int vph = (sv == 0 ? vcnt[0]++ : sv == 1 ? vcnt[1]++ : vcnt[2]++);
                        ok = mbar_wait<true>(BAR(C::B_VFULL + sv), (uint32_t)vph & 1u, abort_flag, flags);
                        if (!(ok = __all_sync(0xffffffffu, ok))) break;
                        tc_fence_after();
                        const uint32_t a_tmem = tmem + C::COL_S + (uint32_t)(sb * BN);
#pragma unroll
                        for (int kk8 = 0; kk8 < BN / 8; ++kk8) {
                            // V^T: this CTA's 64 d rows, 32 keys per 128-byte row, key chunks 8 KB apart
                            const int kc = kk8 / 4, kk = kk8 % 4;
                            const uint64_t b = vdesc0 + (uint64_t)((sv * C::VT + kc * C::VTCH + kk * 32) >> 4);
                            mma_tf32_ts_pair(tmem + C::COL_O, a_tmem + 8 * kk8, b, id_pv, (j > 0 || kk8 > 0) ? 1u : 0u);
                        }
                        mma_commit_pair(BAR(C::B_ODONE + sb));
                        mma_commit_pair(BAR(C::B_VEMPTY + sv));
                    }
                    if (!ok) break;
                    mma_commit_pair(BAR(C::B_OFINAL));
                    fv += w.nblk + C::OSLOTS;
                }
                g0 += w.nblk;
                ++t;
            }
            if (!ok && lane == 0) st_cluster_u32(peer_abort, 1u);
            mma_commit_pair(BAR(C::B_FIN));     // both CTAs see when this warp's products are done
        }
    } else if (warp >= kPfVWarp0 && warp < kPfVWarp0 + 4) {
        // ================================================================ Q and V^T
        // Each thread rounds its query row of the Q buffer to nearest TF32 in place (its eight
        // 16-byte chunks at their swizzled places, so a quarter-warp touches eight distinct banks).
        // Each V half arrives as 2 d chunks x 128 key rows (swizzled like K) and is rewritten in
        // place as V^T: 4 key chunks x 64 d rows, with the diagonal 4x4-block map of prefill_tc.cuh,
        // which keeps both the 16-byte loads and the 16-byte stores free of bank conflicts.
        const int wv = warp - kPfVWarp0;                      // 0..3
        constexpr int DH = D / 2;                             // this CTA's d columns of V
        constexpr int PER = (BN / 4) * (DH / 4) / 128;        // 4x4 blocks per thread per tile
        static_assert(PER == 4, "V transposer work split");
        auto blk = [&](int it, int& aa, int& dq) {
            const int q = lane & 7;
            const int c = it * 16 + wv * 4 + (lane >> 3);    // quarter-warp's (s, ah, dh)
            const int rest = c >> 3;
            aa = 8 * (rest % (BN / 32)) + q;                 // key quad 0..31
            dq = 8 * (rest / (BN / 32)) + (q ^ (c & 7));     // d quad 0..15
        };
        auto staged = [](int key, int dq) -> int {
            return (dq >> 3) * C::VCH + key * 128 + (((dq & 7) ^ (key & 7)) << 4);
        };
        const uint32_t l_qready = LEAD(C::B_QREADY);
        bool ok = true;
        int gb = 0, t = 0;                                   // V-ring fills, items with keys
        const int qr = wv * 32 + lane;                       // query row of the tile
        for (int k = 0; ok; ++k) {
            const int u = pp_item(k);
            if (u >= n_work) break;
            const PpWork w = work(u);
            if (w.nblk == 0) continue;
            {   // ---- query tile: rounded to nearest TF32 in place
                // the four warps decide together, so none is left waiting at the V barrier below
                const bool okq = mbar_wait(BAR(C::B_QLOADED), (uint32_t)t & 1u, abort_flag, flags);
                if (named_barrier_or(3, 128, !okq || *abort_flag)) { ok = false; break; }
#pragma unroll 1
                for (int c = 0; c < C::NCH; ++c) {
                    unsigned char* row = smem + C::OFF_Q + c * C::QCH + qr * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4* p = reinterpret_cast<uint4*>(row + ((j ^ (qr & 7)) << 4));
                        uint4 x = *p;
                        x.x = tf32_round_bits(x.x);
                        x.y = tf32_round_bits(x.y);
                        x.z = tf32_round_bits(x.z);
                        x.w = tf32_round_bits(x.w);
                        *p = x;
                    }
                }
                fence_proxy_async();          // generic-proxy stores -> tensor-core reads
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(l_qready);
                ++t;
            }
            // ---- V blocks of this item
            for (int j = 0; j < w.nblk; ++j, ++gb) {
                const int s = gb % C::NV;
                unsigned char* vt = smem + C::OFF_V + s * C::VT;
                const int kvalid = w.n_kv - j * BN;
                const bool loaded =
                    mbar_wait(BAR(C::B_VLOADED + s), (uint32_t)(gb / C::NV) & 1u, abort_flag, flags);
                float4 x[PER][4];
#pragma unroll
                for (int it = 0; it < PER && loaded; ++it) {
                    int aa, dq;
                    blk(it, aa, dq);
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
                        x[it][rr] = *reinterpret_cast<const float4*>(vt + staged(aa * 4 + rr, dq));
                }
                if (GUARD && kvalid < BN) {   // rows past the sequence (e.g. unwritten cache rows) -> 0
#pragma unroll
                    for (int it = 0; it < PER; ++it) {
                        int aa, dq;
                        blk(it, aa, dq);
#pragma unroll
                        for (int rr = 0; rr < 4; ++rr)
                            if (aa * 4 + rr >= kvalid) x[it][rr] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                if (named_barrier_or(2, 128, !loaded || *abort_flag)) { ok = false; break; }
#pragma unroll
                for (int it = 0; it < PER; ++it) {
                    int aa, dq;
                    blk(it, aa, dq);
                    const int kc = aa >> 3;                  // 32-key chunk of the V^T row
                    const float4 c0 = x[it][0], c1 = x[it][1], c2 = x[it][2], c3 = x[it][3];
                    auto rb = [](float v) { return tf32_round_bits(__float_as_uint(v)); };
                    const uint4 wr[4] = {make_uint4(rb(c0.x), rb(c1.x), rb(c2.x), rb(c3.x)),
                                         make_uint4(rb(c0.y), rb(c1.y), rb(c2.y), rb(c3.y)),
                                         make_uint4(rb(c0.z), rb(c1.z), rb(c2.z), rb(c3.z)),
                                         make_uint4(rb(c0.w), rb(c1.w), rb(c2.w), rb(c3.w))};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int d = dq * 4 + i;
                        const int off = kc * C::VTCH + d * 128 + (((aa & 7) ^ (d & 7)) << 4);
                        *reinterpret_cast<uint4*>(vt + off) = wr[i];
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(LEAD(C::B_VFULL + s));
            }
            if (!ok) break;
            gb += C::OSLOTS;                                 // output staging fills: the epilogue's
        }
        if (!ok) st_cluster_u32(peer_abort, 1u);
    } else {
        // ================================================================ softmax / epilogue
        const int quad = warp & 3;                       // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;                  // query row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        bool ok = true;
        int g0 = 0, t = 0, fv = 0;     // blocks, items with keys, V-ring fills passed
        for (int k = 0; ok; ++k) {
            const int u = pp_item(k);
            if (u >= n_work) break;
            const PpWork w = work(u);
            const int qi = w.q0 + r;
            if (w.nblk == 0) {      // no key is visible to any row of this tile: padding -> zeros
                if (qi < S && in_bounds(((int64_t)w.b * S + qi) * q_row + (int64_t)w.h * D, (int64_t)B * S * q_row, flags)) {
                    float4* op = reinterpret_cast<float4*>(o + ((int64_t)w.b * S + qi) * q_row + (int64_t)w.h * D);
#pragma unroll
                    for (int e = 0; e < D / 4; ++e) __stcs(op + e, make_float4(0.f, 0.f, 0.f, 0.f));
                }
                continue;
            }
            float m_run = -INFINITY, l_run = 0.0f;
            const int key_lim = causal ? min(w.p0 + qi + 1, w.n_kv) : w.n_kv;   // keys visible to this row
            for (int j = 0; j < w.nblk; ++j) {
                const int gb = g0 + j, sb = gb % C::NSBUF;
                ok = mbar_wait(BAR(C::B_SFULL + sb), (uint32_t)(gb / C::NSBUF) & 1u, abort_flag, flags);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;   // warp-uniform before TMEM access
                tc_fence_after();
                const uint32_t s_col = lane_base + C::COL_S + (uint32_t)(sb * BN);
                // S is read out of TMEM twice in 32-column chunks, with the chunk loops rolled: the
                // code stays small (fewer instruction-cache misses) and no more than one chunk of
                // scores is live at a time.
                const int nvis = min(max(key_lim - j * BN, 0), BN);     // visible keys of this block
                const bool masked = __any_sync(0xffffffffu, nvis < BN);
                // pass 1: the block's row maximum (columns past nvis left out)
                float mx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t wv[32];
                    tmem_ld32(s_col + 32 * c, wv);
                    tmem_wait_ld();
                    if (masked) {
                        const int lim = nvis - 32 * c;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            mx[e & 7] = fmaxf(mx[e & 7], e < lim ? __uint_as_float(wv[e]) : -INFINITY);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(wv[e]));
                    }
                }
                // S holds raw q.k; scores in the exponent's units are s * scale*log2(e) (> 0, so the
                // maximum commutes with the scaling)
                const float m_blk = scale_log2 * fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                // m_use is finite: every row of an item with keys sees at least key 0
                const bool need = m_blk > m_run + kLazyRescale;
                const float m_use = need ? m_blk : m_run;
                const float alpha = need ? fast_exp2(m_run - m_blk) : 1.0f;
                // pass 2: p = 2^(s*c - m), truncated to TF32 as the tensor core reads it, written back
                // over S; the row sum is taken over exactly those values in eight partial sums (column
                // e into sum e & 7), two columns at a time through the packed f32x2 FMA and add (each
                // lane rounded as the scalar operation; packed sum k holds partial sums 2k and 2k+1)
                uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
                const uint64_t sl2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_use, -m_use);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t wv[32];
                    tmem_ld32(s_col + 32 * c, wv);
                    tmem_wait_ld();
                    if (masked) {
                        const int lim = nvis - 32 * c;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e >= lim) wv[e] = __float_as_uint(-INFINITY);     // 2^-inf = +0
                    }
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(wv[e]), __uint_as_float(wv[e + 1])), sl2, nm2), t0, t1);
                        wv[e] = __float_as_uint(fast_exp2(t0)) & 0xFFFFE000u;
                        wv[e + 1] = __float_as_uint(fast_exp2(t1)) & 0xFFFFE000u;
                        ls2[(e & 7) >> 1] =
                            f2_add(ls2[(e & 7) >> 1], f2_pack(__uint_as_float(wv[e]), __uint_as_float(wv[e + 1])));
                    }
                    tmem_st32(s_col + 32 * c, wv);
                }
                float ls[8];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) f2_unpack(ls2[k2], ls[2 * k2], ls[2 * k2 + 1]);
                const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                l_run = l_run * alpha + lsum;
                m_run = m_use;
                tmem_wait_st();
                if (j > 0 && __any_sync(0xffffffffu, need)) {
                    // O holds blocks < j once PV_{gb-1} completes; scale it by alpha (parity wait
                    // exact as in prefill_tc.cuh)
                    ok = mbar_wait(BAR(C::B_ODONE + (gb - 1) % C::NSBUF), (uint32_t)((gb - 1) / C::NSBUF) & 1u,
                                   abort_flag, flags);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t wv[32];
                        tmem_ld32(lane_base + C::COL_O + 32 * c, wv);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) wv[e] = __float_as_uint(__uint_as_float(wv[e]) * alpha);
                        tmem_st32(lane_base + C::COL_O + 32 * c, wv);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(LEAD(C::B_PREADY + sb));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            ok = mbar_wait(BAR(C::B_OFINAL), (uint32_t)t & 1u, abort_flag, flags);
            if (!(ok = __all_sync(0xffffffffu, ok))) break;
            tc_fence_after();
            const bool live = qi < w.len && l_run > 0.0f;
            const float inv = live ? 1.0f / l_run : 0.0f;
            const int fs = fv + w.nblk;                          // first staging fill
#pragma unroll 1
            for (int i = 0; ok && i < C::OSLOTS; ++i) {
                ok = mbar_wait(BAR(C::B_VLOADED + (fs + i) % C::NV), (uint32_t)((fs + i) / C::NV) & 1u, abort_flag,
                               flags);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                unsigned char* stage = smem + C::OFF_V + ((fs + i) % C::NV) * C::VT;
#pragma unroll 1
                for (int cc = 0; cc < C::OCH; ++cc) {
                    const int c = i * C::OCH + cc;               // column chunk of O
                    unsigned char* dst = stage + cc * C::QCH;
                    uint32_t wv[32];
                    tmem_ld32(lane_base + C::COL_O + 32 * c, wv);
                    tmem_wait_ld();
                    if (GUARD && !live) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) wv[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        *reinterpret_cast<float4*>(dst + r * 128 + (((e & 7) ^ (r & 7)) << 4)) =
                            make_float4(__uint_as_float(wv[4 * e]) * inv, __uint_as_float(wv[4 * e + 1]) * inv,
                                        __uint_as_float(wv[4 * e + 2]) * inv, __uint_as_float(wv[4 * e + 3]) * inv);
                }
                fence_proxy_async();                             // generic stores -> TMA reads
                mbar_arrive(BAR(C::B_OSTAGED + i));
            }
            if (!ok) break;
            fv += w.nblk + C::OSLOTS;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(LEAD(C::B_OFREE));   // O may be overwritten
            g0 += w.nblk;
            ++t;
        }
        if (!ok) st_cluster_u32(peer_abort, 1u);
    }

    // ---------------------------------------------------------------- teardown
    // Both issuers' last commits reach both CTAs once all their products are done; after that and
    // a cluster-wide barrier no CTA is touched by the other any more.
    if (warp == 1 && lane == 0) mbar_drain(BAR(C::B_FIN), 0u, kWaitLimitNs);
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kPfTmemCols);
    }
}

}  // namespace rkv
