#pragma once
// prefill_tc.cuh -- fused flash-style prefill on the 5th-generation tensor core (sm_103a).
//
// Semantics: trueno-gpu 0.4.11 src/memory/resident/attention.rs,
// fn batched_multihead_attention_optimized (interleaved [seq, n_heads*head_dim]
// in and out, scale 1/sqrt(head_dim)) and trustformers-core 0.2.0
// src/gpu_ops/cuda/oxicuda/attention.rs, fn attention_prefill_gpu_to_gpu
// (causal: query i sees keys 0..=i; per head: scaled GEMM, causal softmax,
// GEMM).  Here all of it is one kernel: heads are read in place, the score
// tile never leaves tensor memory, and softmax is online (base 2).
//
// The kernel is persistent: one CTA per SM walks a static list of work items (a
// 128-query tile of one (batch, head)), heaviest causal tiles first, dealt in rounds
// that alternate direction.  Rings, TMEM buffers and barrier phases run on across
// items, so one item's prologue (Q load) and epilogue (O store) overlap the tensor-core
// work of its neighbours.  Warp roles:
//   warp 0       K producer (one thread): TMA (cp.async.bulk.tensor, 128-byte
//                swizzle) of BN x D tiles into an NK-stage ring that carries each
//                item's query tile ahead of its key tiles; it also prefetches the
//                next item's query tile into L2.
//   warp 11      V producer (one thread): V tiles into an NV-stage ring, followed per
//                item by output staging slots that the epilogue fills with O / l and
//                this thread stores to the output by TMA.
//   warp 1       QK^T issuer (one thread) and TMEM owner: per key block
//                  S_j = Q . K_j^T   tcgen05.mma kind::tf32, A = Q from TMEM
//                S goes to NSBUF TMEM buffers, so QK^T runs up to NSBUF blocks
//                ahead of the softmax.
//   warp 10      PV issuer (one thread):  O += P_j . V_j, A = P from TMEM.
//   warps 2-5    softmax / epilogue, one thread per query row (TMEM lane): per
//                block: S row from TMEM, mask, row max, lazy rescale (O is
//                rescaled only when the running max grows by more than 2^8),
//                p = 2^(s*scale*log2e - m) truncated to TF32 and written back over
//                S; per item: O / l written to the staging slots (swizzled like the
//                TMA box, conflict-free).
//   warps 6-9    Q and V^T: per item, the query tile goes from the K ring through
//                registers (rounded to nearest TF32) into TMEM by tcgen05.st; tcgen05
//                kind::tf32 reads B only K-major, so each V tile is transposed in
//                shared memory (4x4 blocks through registers, rounded to nearest TF32,
//                conflict-free 16-byte loads and stores, 128-byte swizzle).
// Q, K and V stay f32 in memory.  The tensor core reads an f32 operand as TF32 by dropping
// its low 13 bits: K is used as loaded (truncated), Q and V are rounded to nearest on their
// way through registers (half the worst-case error of truncation, no bias), P is truncated
// and the row sum is taken over exactly the truncated values.
// Every mbarrier wait is time-bounded (see rkv_internal.cuh); a CTA that gives
// up unwinds: it drains its own copies in flight, lets issued MMAs finish and
// frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

constexpr int kPfBM = 128;                    // query rows per CTA (TMEM lanes)
constexpr int kPfThreads = 384;               // 12 warps
constexpr int kPfPvWarp = 10;                 // PV issuer
constexpr int kPfVWarp0 = 6;                  // first V transposer warp
constexpr int kPfVProdWarp = 11;              // V producer and output stores
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
    static constexpr uint32_t K_ATOM = D >= 32 ? 1024 : 512; // 8 rows x swizzle span
    // Each item's query tile travels through the K ring ahead of its K tiles, as QSLOTS
    // fills of BN rows (same box as a K tile).  With paired slots the query fills take one
    // aligned slot pair, so their 128 rows sit at a uniform stride like an MMA operand.
    static constexpr int QSLOTS = kPfBM / BN;
    static_assert(QSLOTS <= NK && (!KPAIR || QSLOTS == 2), "query fills in the K ring");
    // Each item's output tile (kPfBM x D) is staged in OSLOTS V-ring slots, each holding
    // OCH column chunks of CH floats for all kPfBM rows (swizzled like the TMA box).
    static constexpr int OSLOTS = kPfBM / BN;
    static constexpr int OCH = NCH / OSLOTS;
    static_assert(OSLOTS < NV && OSLOTS * OCH == NCH && OCH * kPfBM * CH * 4 == TILE, "output staging");
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
    //           p_ready[NSBUF], o_done[NSBUF], o_final, q_free, o_free, drain, drain_pv, q_ready
    static constexpr int NBAR = 2 * NK + 3 * NV + 3 * NSBUF + 6;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;     // tmem base, abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM = (SMEM_USED + 1024 > kPfMinSmem ? SMEM_USED + 1024 : kPfMinSmem);
    static_assert(SMEM <= 227 * 1024, "prefill shared memory budget");
    static_assert(kColS + NSBUF * S_BUF <= (int)kPfTmemCols && kColO + PV_SPLIT * D <= kColS && D <= 128,
                  "TMEM budget");
};

struct PfBars {
    uint32_t k_full, k_empty, v_full, v_empty, v_loaded, s_full, p_ready, o_done, o_final, q_free, o_free,
        drain, drain_pv, q_ready;
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
    b.q_free = b.o_final + 8;
    b.o_free = b.q_free + 8;
    b.drain = b.o_free + 8;
    b.drain_pv = b.drain + 8;
    b.q_ready = b.drain_pv + 8;
    return b;
}

// One work item: a 128-query tile of one (batch, head).  Query i of the sequence sits at
// key position p0 + i; the sequence has n_kv keys (p0 + len, at most the key capacity).
struct PfWork {
    int b, h, g, q0, len, p0, n_kv, nblk;
};

// Where the keys and values of (batch b, kv head g) live for the tensor copies:
// coordinates (g * xg + d, key, b * zb + g * zg).  Interleaved activations [B, S, Hk*D]:
// (xg, zb, zg) = (D, 1, 0); the cache [B, Hk, max_len, D]: (0, Hk, 1).
struct PfKv {
    int xg, zb, zg, cap;            // cap: key capacity (S, or the cache's max_len)
    const int* start;               // per-sequence key offset p0 (device), NULL -> 0
};

// Work items are numbered heaviest causal tiles first: u -> (tile n_qtiles-1-u/BH, bh = u%BH).
template <int D>
__device__ __forceinline__ PfWork pf_work(int u, int B, int H, int Hk, int S, int n_qtiles, int causal,
                                          const int* __restrict__ seq_lens, const PfKv& kv) {
    const int BH = B * H;
    PfWork w;
    const int tile = n_qtiles - 1 - u / BH;
    const int bh = u % BH;
    w.b = bh / H;
    w.h = bh % H;
    w.g = w.h / (H / Hk);
    w.q0 = tile * kPfBM;
    w.len = seq_lens ? min(max(__ldg(seq_lens + w.b), 0), S) : S;
    w.p0 = kv.start ? min(max(__ldg(kv.start + w.b), 0), kv.cap) : 0;
    w.n_kv = min(w.p0 + w.len, kv.cap);
    const int kv_end = w.q0 >= w.len ? 0 : (causal ? min(w.n_kv, w.p0 + w.q0 + kPfBM) : w.n_kv);
    w.nblk = (kv_end + PfCfg<D>::BN - 1) / PfCfg<D>::BN;
    return w;
}

// The k-th work item of this CTA.  Items are dealt in rounds of gridDim.x, every other
// round in reverse CTA order, so the heavy-first costs even out across CTAs.
__device__ __forceinline__ int pf_item(int k) {
    const int G = (int)gridDim.x;
    return k * G + ((k & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// GUARD: some keys or queries of a tile may lie past a sequence's valid part (per-sequence
// lengths, or keys read from a cache whose rows past the sequence may hold anything).  Only
// then are V rows past the sequence zeroed and padded output rows forced to zero; without
// it every loaded row is inside the tensors (rows past them are zero-filled by the copy
// engine and clipped on store) and the kernel carries none of that code.
// FILL: the launch is followed by a programmatic dependent (the cache fill, kv_scatter.cu),
// which this kernel releases at once so that it runs beside the attention, in the registers and
// shared memory the prefill leaves free on each SM.  For that the FILL variant at D = 128 is
// held to kPfFillRegs registers a thread: 384 x 144 + the fill's 256 x 40 fill the 64K
// register file (at D <= 64 the kernel needs more, and the fill runs in what is left).
constexpr int kPfFillRegs = 144;
template <int D, bool GUARD, bool FILL>
__global__ void __maxnreg__(FILL && D == 128 ? kPfFillRegs : 65536 / kPfThreads / 8 * 8)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                  float* __restrict__ o,
                  int B, int S, int H, int Hk, int causal, const int* __restrict__ seq_lens, float scale_log2,
                  int n_qtiles, int n_work, const PfKv kv, unsigned int* __restrict__ flags) {
    using C = PfCfg<D>;
    constexpr int BN = C::BN;
    static_assert(!(FILL && GUARD), "the fused cache fill is built for whole sequences only");
    if (FILL) griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    const PfBars bar = pf_bars<C::NK, C::NV, C::NSBUF>(smem_addr(smem + C::OFF_BAR));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t q_row = (int64_t)H * D;
    auto work = [&](int u) { return pf_work<D>(u, B, H, Hk, S, n_qtiles, causal, seq_lens, kv); };

    if ((seq_lens || kv.start) && blockIdx.x == 0) {     // report clamped lengths once per launch
        for (int i = threadIdx.x; i < B; i += blockDim.x) {
            const int l = seq_lens ? __ldg(seq_lens + i) : S;
            const int p = kv.start ? __ldg(kv.start + i) : 0;
            if (l > S || (int64_t)max(p, 0) + min(max(l, 0), S) > kv.cap) atomicOr(flags, RKV_FLAG_LEN_CLAMPED);
            if (l < 0 || p < 0) atomicOr(flags, RKV_FLAG_NEGATIVE_INPUT);
        }
    }

    // ------------------------------------------------------------------ setup
    // Thread 0 initialises the barriers and is also the K producer: it issues the first item's
    // query tile and first key tiles straight away (the barriers are fresh, no slot to wait
    // for), so they are in flight while tensor memory is allocated and the CTA synchronises.
    int k_first = -1, k_pre = 0;                   // (thread 0) that item and its fills issued
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
        mbar_init(bar.q_free, 1);
        mbar_init(bar.o_free, 128);
        mbar_init(bar.drain, 1);
        mbar_init(bar.drain_pv, 1);
        mbar_init(bar.q_ready, 128);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_o);
        for (int k = 0;; ++k) {
            const int u = pf_item(k);
            if (u >= n_work) break;
            const PfWork w = work(u);
            if (w.nblk == 0) continue;
            k_first = k;
            k_pre = min(C::NK, C::QSLOTS + w.nblk);
            for (int f = 0; f < k_pre; ++f) {          // fill f of the ring: query tile, then keys
                const uint32_t full = bar.k_full + 8 * f;
                mbar_arrive_expect_tx(full, C::TILE);
                const int j = f - C::QSLOTS;
                const bool qfill = j < 0;
                const void* map = qfill ? static_cast<const void*>(&tm_q) : static_cast<const void*>(&tm_k);
                const int x0 = qfill ? w.h * D : w.g * kv.xg;
                const int y0 = qfill ? w.q0 + f * BN : j * BN;
                const int z0 = qfill ? w.b : w.b * kv.zb + w.g * kv.zg;
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(smem_addr(smem + C::OFF_K) + C::koff(f, c), map, x0 + c * C::CH, y0, z0, full);
            }
            break;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Every role walks the same item sequence and numbers key blocks with one running
    // counter (g) across items, so ring slots and barrier phases continue from item to
    // item.  Items without visible keys use no barrier at all.
    if (warp == 0) {
        // ================================================================ K producer
        // lane 0: per item [pad] the query tile (QSLOTS fills) then one K tile per block, by TMA.
        // With paired slots the query fills must start on an even fill; an empty pad fill (a
        // plain arrival, no data) restores that after an odd block count.
        if (lane == 0) {
            int gs = k_pre;               // fills of the K ring so far (the first ones issued at setup)
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int u = pf_item(k);
                if (u >= n_work) break;
                const PfWork w = work(u);
                if (w.nblk == 0) continue;
                {                   // the next item's query tile -> L2, ahead of its own copy
                    const int un = pf_item(k + 1);
                    if (un < n_work) {
                        const PfWork wn = work(un);
#pragma unroll
                        for (int i = 0; i < C::QSLOTS; ++i)
#pragma unroll
                            for (int c = 0; c < C::NCH; ++c)
                                tma_prefetch_l2_3d(&tm_q, wn.h * D + c * C::CH, wn.q0 + i * BN, wn.b);
                    }
                }
                const bool first = k == k_first;
                const bool pad = !first && C::KPAIR && (gs & 1);
                constexpr int nq = C::QSLOTS;
                for (int j = first ? k_pre - nq : -nq - (pad ? 1 : 0); j < w.nblk; ++j) {
                    const int s = gs % C::NK;
                    if (!(ok = mbar_wait(bar.k_empty + 8 * s, ((uint32_t)(gs / C::NK) & 1u) ^ 1u, abort_flag, flags)))
                        break;
                    const uint32_t full = bar.k_full + 8 * s;
                    ++gs;
                    if (j < -nq) {          // pad fill
                        mbar_arrive(full);
                        continue;
                    }
                    mbar_arrive_expect_tx(full, C::TILE);
                    const bool qfill = j < 0;
                    const void* map = qfill ? static_cast<const void*>(&tm_q) : static_cast<const void*>(&tm_k);
                    const int x0 = qfill ? w.h * D : w.g * kv.xg;
                    const int y0 = qfill ? w.q0 + (j + nq) * BN : j * BN;
                    const int z0 = qfill ? w.b : w.b * kv.zb + w.g * kv.zg;
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d(smem_addr(smem + C::OFF_K) + C::koff(s, c), map, x0 + c * C::CH, y0, z0, full);
                }
            }
            if (*abort_flag) {   // unwinding: let issued copies land
                for (int f = max(0, gs - C::NK); f < gs; ++f)
                    mbar_drain(bar.k_full + 8 * (f % C::NK), (uint32_t)(f / C::NK) & 1u, 100000000ull);
            }
        }
    } else if (warp == kPfVProdWarp) {
        // ================================================================ V producer / O stores
        // lane 0: per item one V tile per block by TMA, then OSLOTS output staging fills: no
        // data, the slot is handed (plain arrival on v_loaded) to the epilogue, which writes
        // O / l there and arrives on v_full.  This thread then stores the staged tile to the
        // output by TMA and, once the copy engine has read it, releases the slots.  It does
        // so before the first later fill that reuses one of them (or at the end).
        if (lane == 0) {
            int gs = 0;                   // fills of the V ring so far
            bool ok = true;
            int pend = -1;                // first staging fill not yet stored (-1: none)
            PfWork pw{};                  // its item
            auto flush = [&]() -> bool {
                for (int i = 0; i < C::OSLOTS; ++i)
                    if (!mbar_wait(bar.v_full + 8 * ((pend + i) % C::NV), (uint32_t)((pend + i) / C::NV) & 1u,
                                   abort_flag, flags))
                        return false;
                for (int i = 0; i < C::OSLOTS; ++i) {
                    const uint32_t src = smem_addr(smem + C::OFF_V) + ((pend + i) % C::NV) * C::TILE;
#pragma unroll
                    for (int cc = 0; cc < C::OCH; ++cc)
                        tma_store_3d(&tm_o, src + cc * (kPfBM * C::CH * 4), pw.h * D + (i * C::OCH + cc) * C::CH,
                                     pw.q0, pw.b);
                }
                bulk_commit();
                bulk_wait_read_all();
                for (int i = 0; i < C::OSLOTS; ++i) mbar_arrive(bar.v_empty + 8 * ((pend + i) % C::NV));
                pend = -1;
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int u = pf_item(k);
                if (u >= n_work) break;
                const PfWork w = work(u);
                if (w.nblk == 0) continue;
                for (int j = 0; j < w.nblk + C::OSLOTS; ++j) {
                    if (pend >= 0 && gs >= pend + C::NV && !(ok = flush())) break;
                    const int s = gs % C::NV;
                    if (!(ok = mbar_wait(bar.v_empty + 8 * s, ((uint32_t)(gs / C::NV) & 1u) ^ 1u, abort_flag, flags)))
                        break;
                    const uint32_t full = bar.v_loaded + 8 * s;
                    if (j >= w.nblk) {      // output staging fill
                        if (j == w.nblk) { pend = gs; pw = w; }
                        ++gs;
                        mbar_arrive(full);
                        continue;
                    }
                    ++gs;
                    mbar_arrive_expect_tx(full, C::TILE);
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d(smem_addr(smem + C::OFF_V) + s * C::TILE + c * BN * C::CH * 4, &tm_v,
                                    w.g * kv.xg + c * C::CH, j * BN, w.b * kv.zb + w.g * kv.zg, full);
                }
            }
            if (ok && pend >= 0) ok = flush();
            bulk_wait_all();                  // output stores complete before the CTA exits
            if (*abort_flag) {   // unwinding: let issued copies land
                for (int f = max(0, gs - C::NV); f < gs; ++f)
                    mbar_drain(bar.v_loaded + 8 * (f % C::NV), (uint32_t)(f / C::NV) & 1u, 100000000ull);
            }
        }
    } else if (warp == 1 || warp == kPfPvWarp) {
        // ================================================================ MMA issuers
        // Two warps issue: warp 1 the QK^T MMAs, warp 10 the PV MMAs.  Each walks its loop as a
        // whole warp (every value in it is warp-uniform), waits are decided by the warp together,
        // one elected lane executes each MMA and commit, and lane 0 makes the plain arrivals.
        {
            const bool qk_role = warp == 1;
            constexpr uint32_t id_qk = idesc_tf32(kPfBM, BN, false);
            constexpr uint32_t id_qk2 = idesc_tf32(kPfBM, 2 * BN, false);
            constexpr uint32_t id_pv = idesc_tf32(kPfBM, D, false);
            bool ok = true;
            int issued_any = 0, g0 = 0, t = 0;   // t: items with keys so far
            int f = 0;                           // K-ring fills consumed (QK^T issuer)
            int fv = 0;                          // V-ring fills passed (PV issuer)
            // Descriptors are built once; a k step or ring stage only adds its byte offset
            // (>> 4) to the start-address field, which cannot carry out of it (shared
            // addresses are below 2^18).
            const uint64_t kdesc0 = smem_desc(smem_addr(smem + C::OFF_K), 16, C::K_ATOM, C::K_SWIZZLE);
            const uint64_t vdesc0 = smem_desc(smem_addr(smem + C::OFF_V), 16, 1024, kSwizzle128B);
            for (int k = 0; ok; ++k) {
                const int u = pf_item(k);
                if (u >= n_work) break;
                const PfWork w = work(u);
                if (w.nblk == 0) continue;
                if (qk_role) {
                    // K-ring fills of this item: [pad] query tile (QSLOTS) then one per key block
                    if (C::KPAIR && (f & 1)) {      // pad fill: nothing to read, hand it back
                        ok = mbar_wait(bar.k_full + 8 * (f % C::NK), (uint32_t)(f / C::NK) & 1u, abort_flag, flags);
                        if (!(ok = __all_sync(0xffffffffu, ok))) break;
                        if (lane == 0) mbar_arrive(bar.k_empty + 8 * (f % C::NK));
                        ++f;
                    }
                    // The Q/V^T warps read the item's query tile out of the K ring, round it and
                    // write it into TMEM columns kColQ.. (after the previous item's QK^T MMAs,
                    // committed to q_free, are done reading them).  Once they have, the query
                    // slots are handed back to the K producer.
                    ok = mbar_wait(bar.q_ready, (uint32_t)t & 1u, abort_flag, flags);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
                    if (lane == 0)
                        for (int i = 0; i < C::QSLOTS; ++i) mbar_arrive(bar.k_empty + 8 * ((f + i) % C::NK));
                    f += C::QSLOTS;
                    // S of block gb goes to buffer gb % NSBUF.  Paired blocks (D = 128: fill f
                    // even, adjacent buffers) share one N = 2*BN chain.  Before QK overwrites a
                    // buffer, the PV that read P from it (block gb - NSBUF) must have finished.
                    // The wait is exact: PV_{gb-2*NSBUF} completed before QK_{gb-NSBUF} was
                    // issued, and PV_gb cannot have started (it needs S_gb).
                    for (int j = 0; ok && j < w.nblk;) {
                        const int gb = g0 + j, fb = f + j;
                        const int nb = (C::KPAIR && (fb & 1) == 0 && gb % C::NSBUF != C::NSBUF - 1 && j + 1 < w.nblk)
                                           ? 2 : 1;
                        for (int i = 0; ok && i < nb; ++i) {
                            if (gb + i >= C::NSBUF)
                                ok = mbar_wait(bar.o_done + 8 * ((gb + i) % C::NSBUF),
                                               (uint32_t)((gb + i - C::NSBUF) / C::NSBUF) & 1u, abort_flag, flags);
                            if (ok)
                                ok = mbar_wait(bar.k_full + 8 * ((fb + i) % C::NK), (uint32_t)((fb + i) / C::NK) & 1u,
                                               abort_flag, flags);
                        }
                        if (!(ok = __all_sync(0xffffffffu, ok))) break;
                        tc_fence_after();
                        const int s = fb % C::NK;
                        const uint32_t d_tmem = tmem + kColS + (uint32_t)((gb % C::NSBUF) * C::S_BUF);
#pragma unroll
                        for (int kk8 = 0; kk8 < D / 8; ++kk8) {
                            const int c = kk8 / (C::CH / 8), kk = kk8 % (C::CH / 8);
                            const uint64_t bdesc = kdesc0 + (uint64_t)((C::koff(s, c) + kk * 32) >> 4);
                            mma_tf32_ts(d_tmem, tmem + kColQ + 8 * kk8, bdesc, nb == 2 ? id_qk2 : id_qk,
                                        kk8 > 0 ? 1u : 0u);
                        }
                        for (int i = nb - 1; i >= 0; --i) mma_commit(bar.s_full + 8 * ((gb + i) % C::NSBUF));
                        for (int i = 0; i < nb; ++i) mma_commit(bar.k_empty + 8 * ((fb + i) % C::NK));
                        issued_any = 1;
                        j += nb;
                    }
                    if (!ok) break;
                    f += w.nblk;
                    mma_commit(bar.q_free);    // all QK^T of this item done: Q columns reusable
                } else {
                    // O is reused item after item: PV of a new item starts (accumulate = 0)
                    // only after the epilogue has read the previous item's O.
                    if (t > 0) ok = mbar_wait(bar.o_free, (uint32_t)(t - 1) & 1u, abort_flag, flags);
                    ok = __all_sync(0xffffffffu, ok);
                    for (int j = 0; ok && j < w.nblk; ++j) {
                        // O += P_gb V_gb
                        const int gb = g0 + j, vf = fv + j;
                        const int sv = vf % C::NV, sb = gb % C::NSBUF;
                        ok = mbar_wait(bar.p_ready + 8 * sb, (uint32_t)(gb / C::NSBUF) & 1u, abort_flag, flags);
                        if (ok) ok = mbar_wait(bar.v_full + 8 * sv, (uint32_t)(vf / C::NV) & 1u, abort_flag, flags);
                        if (!(ok = __all_sync(0xffffffffu, ok))) break;
                        tc_fence_after();
                        const uint64_t vd = vdesc0 + (uint64_t)(sv * (C::TILE >> 4));
                        const uint32_t a_tmem = tmem + kColS + (uint32_t)(sb * C::S_BUF);
                        const uint32_t first = j > 0 ? 1u : 0u;
#pragma unroll
                        for (int kk8 = 0; kk8 < BN / 8; ++kk8) {
                            // V^T tile: rows = d, 32 keys per 128-byte row, key chunks D*128 bytes apart
                            const uint64_t bdesc = vd + (uint64_t)(((kk8 / 4) * (D * 128) + (kk8 % 4) * 32) >> 4);
                            const int part = kk8 % C::PV_SPLIT;
                            mma_tf32_ts(tmem + kColO + part * D, a_tmem + 8 * kk8, bdesc, id_pv,
                                        kk8 >= C::PV_SPLIT ? 1u : first);
                        }
                        mma_commit(bar.o_done + 8 * sb);
                        mma_commit(bar.v_empty + 8 * sv);
                        issued_any = 1;
                    }
                    if (!ok) break;
                    mma_commit(bar.o_final);
                    fv += w.nblk + C::OSLOTS;          // the item's V tiles and output staging fills
                }
                g0 += w.nblk;
                ++t;
            }
            if (!ok && issued_any) {   // unwinding: let issued MMAs finish before TMEM is freed
                const uint32_t dr = qk_role ? bar.drain : bar.drain_pv;
                mma_commit(dr);
                mbar_drain(dr, 0, 100000000ull);
            }
        }
    } else if (warp >= kPfVWarp0 && warp < kPfVWarp0 + 4) {
        // ================================================================ Q and V^T
        // Per item, first the query tile: each thread takes its query row (TMEM lane) out of
        // the K ring (swizzled rows: 16-byte chunk j of row r at j ^ (r & 7), or j ^ ((r >> 1)
        // & 3) with the 64-byte swizzle; conflict-free, eight consecutive rows per quarter-warp),
        // rounds it to nearest TF32 and stores it into TMEM columns kColQ.. of its lane.
        // V tiles arrive by TMA in the same swizzled layout as K (rows = keys).  The
        // transposer rewrites each slot in place as V^T: work item = (key quad aa,
        // d quad dq), a 4x4 block read with four 16-byte loads and written as four
        // 16-byte rows of V^T.  A 16-byte access is served a quarter-warp at a time, so
        // the eight lanes of a quarter-warp must hit eight distinct 16-byte chunks of the
        // 128-byte swizzle, on the loads (chunk (dq ^ key) & 7) and on the stores (chunk
        // (aa ^ d) & 7).  For D >= 32 a quarter-warp takes a diagonal: lane q gets key quad
        // 8*ah + q and d quad 8*dh + (q ^ s), with (s, ah, dh) fixed per quarter-warp and
        // iteration; then both chunk sets are permutations of 0..7.  At D = 16 (64-byte
        // swizzle) a quarter-warp takes 8 consecutive key quads of one d quad.
        const int wv = warp - kPfVWarp0;                      // 0..3
        constexpr int LDQ = D / 4 < 8 ? D / 4 : 8;           // D = 16: lanes along d quads
        constexpr int LAA = 32 / LDQ;                        // D = 16: lanes along key quads
        constexpr int GA = (BN / 4) / LAA;                   // D = 16: lane groups along keys
        constexpr int PER = (BN / 4) * (D / 4) / 128;        // 4x4 blocks per thread per tile
        static_assert((BN / 4) * (D / 4) % 128 == 0 && PER >= 1, "V transposer work split");
        static_assert(D < 32 || (BN % 32 == 0 && D % 32 == 0), "diagonal transposer map");
        const int aa_lo = lane % LAA, dq_lo = lane / LAA;
        // (key quad, d quad) of this thread's it-th block
        auto blk = [&](int it, int& aa, int& dq) {
            if constexpr (D >= 32) {
                const int q = lane & 7;
                const int c = it * 16 + wv * 4 + (lane >> 3);   // quarter-warp's (s, ah, dh)
                const int rest = c >> 3;
                aa = 8 * (rest % (BN / 32)) + q;
                dq = 8 * (rest / (BN / 32)) + (q ^ (c & 7));
            } else {
                const int G = it * 4 + wv;
                aa = (G % GA) * LAA + aa_lo;
                dq = (G / GA) * LDQ + dq_lo;
            }
        };
        // Byte offset of V[key][d] in a TMA-staged tile (box {CH floats, BN keys} per
        // d chunk, swizzled: 16-byte chunk index XOR key bits).
        auto staged = [](int key, int dq) -> int {
            if constexpr (D >= 32)
                return (dq >> 3) * (BN * 128) + key * 128 + (((dq & 7) ^ (key & 7)) << 4);
            else
                return key * 64 + (((dq & 3) ^ ((key >> 1) & 3)) << 4);
        };
        bool ok = true;
        int gb = 0;                                          // V-ring fills passed
        int fk = 0;                                          // K-ring fills passed (as the QK^T issuer)
        int tq = 0;                                          // items with keys so far
        const int qquad = warp & 3;                          // TMEM lane quadrant of this warp
        const int qr = qquad * 32 + lane;                    // query row within the tile
        for (int k = 0; ok; ++k) {
            const int u = pf_item(k);
            if (u >= n_work) break;
            const PfWork w = work(u);
            if (w.nblk == 0) continue;
            // ---- query tile of this item -> TMEM (the previous item's QK^T done with it)
            if (C::KPAIR && (fk & 1)) ++fk;                  // pad fill
            {
                bool okq = true;
                if (tq > 0) okq = mbar_wait(bar.q_free, (uint32_t)(tq - 1) & 1u, abort_flag, flags);
                for (int i = 0; okq && i < C::QSLOTS; ++i)
                    okq = mbar_wait(bar.k_full + 8 * ((fk + i) % C::NK), (uint32_t)((fk + i) / C::NK) & 1u,
                                    abort_flag, flags);
                if (!(ok = __all_sync(0xffffffffu, okq))) break;   // warp-uniform before TMEM access
                tc_fence_after();
                const uint32_t qlane = tmem + ((uint32_t)(qquad * 32) << 16);
                const int sq = fk % C::NK;      // even when paired: the query tile fills a slot pair
#pragma unroll 1
                for (int c = 0; c < C::NCH; ++c) {
                    const unsigned char* row = smem + C::OFF_K + C::koff(sq, c) + qr * (C::CH * 4);
                    if constexpr (C::CH == 32) {
                        uint32_t wv[32];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ (qr & 7)) << 4));
                            wv[4 * j] = tf32_round_bits(x.x);
                            wv[4 * j + 1] = tf32_round_bits(x.y);
                            wv[4 * j + 2] = tf32_round_bits(x.z);
                            wv[4 * j + 3] = tf32_round_bits(x.w);
                        }
                        tmem_st32(qlane + kColQ + 32 * c, wv);
                    } else {                    // D = 16: 64-byte rows, 64-byte swizzle
                        uint32_t wv[16];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ ((qr >> 1) & 3)) << 4));
                            wv[4 * j] = tf32_round_bits(x.x);
                            wv[4 * j + 1] = tf32_round_bits(x.y);
                            wv[4 * j + 2] = tf32_round_bits(x.z);
                            wv[4 * j + 3] = tf32_round_bits(x.w);
                        }
                        tmem_st16(qlane + kColQ, wv);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar.q_ready);
                fk += C::QSLOTS + w.nblk;
                ++tq;
            }
            // ---- V tiles of this item
            for (int j = 0; j < w.nblk; ++j, ++gb) {
                const int s = gb % C::NV;
                unsigned char* vt = smem + C::OFF_V + s * C::TILE;
                // Keys past the sequence get p = 0, but 0 * v is not 0 when v is not finite
                // (cache rows that were never written): those V rows are replaced by zeros.
                const int kvalid = w.n_kv - j * BN;
                const bool loaded = mbar_wait(bar.v_loaded + 8 * s, (uint32_t)(gb / C::NV) & 1u, abort_flag, flags);
                float4 x[PER][4];
#pragma unroll
                for (int it = 0; it < PER && loaded; ++it) {
                    int aa, dq;
                    blk(it, aa, dq);
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
                        x[it][rr] = *reinterpret_cast<const float4*>(vt + staged(aa * 4 + rr, dq));
                }
                if (GUARD && kvalid < BN) {   // the sequence's last block (uniform over the CTA)
#pragma unroll
                    for (int it = 0; it < PER; ++it) {
                        int aa, dq;
                        blk(it, aa, dq);
#pragma unroll
                        for (int rr = 0; rr < 4; ++rr)
                            if (aa * 4 + rr >= kvalid) x[it][rr] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                // every thread has read its blocks: rewrite in place (or leave, all together)
                if (named_barrier_or(2, 128, !loaded || *abort_flag)) { ok = false; break; }
#pragma unroll
                for (int it = 0; it < PER; ++it) {
                    int aa, dq;
                    blk(it, aa, dq);
                    const int kc = aa >> 3;                      // 32-key chunk of the V^T row
                    const float4 c0 = x[it][0], c1 = x[it][1], c2 = x[it][2], c3 = x[it][3];
                    auto rb = [](float x) { return tf32_round_bits(__float_as_uint(x)); };
                    const uint4 wr[4] = {make_uint4(rb(c0.x), rb(c1.x), rb(c2.x), rb(c3.x)),
                                         make_uint4(rb(c0.y), rb(c1.y), rb(c2.y), rb(c3.y)),
                                         make_uint4(rb(c0.z), rb(c1.z), rb(c2.z), rb(c3.z)),
                                         make_uint4(rb(c0.w), rb(c1.w), rb(c2.w), rb(c3.w))};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int d = dq * 4 + i;
                        const int off = kc * (D * 128) + d * 128 + (((aa & 7) ^ (d & 7)) << 4);
                        *reinterpret_cast<uint4*>(vt + off) = wr[i];
                    }
                }
                fence_proxy_async();          // generic-proxy stores -> tensor-core reads
                mbar_arrive(bar.v_full + 8 * s);
            }
            gb += C::OSLOTS;                                 // output staging fills: the epilogue's
        }
    } else {
        // ================================================================ softmax / epilogue
        const int quad = warp & 3;                       // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;                  // query row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        bool ok = true;
        int g0 = 0, t = 0, fv = 0;     // blocks, items with keys, V-ring fills passed
        for (int k = 0; ok; ++k) {
            const int u = pf_item(k);
            if (u >= n_work) break;
            const PfWork w = work(u);
            const int qi = w.q0 + r;
            float4* op = reinterpret_cast<float4*>(o + ((int64_t)w.b * S + qi) * q_row + (int64_t)w.h * D);
            if (w.nblk == 0) {      // no key is visible to any row of this tile: padding -> zeros
                if (qi < S && in_bounds(((int64_t)w.b * S + qi) * q_row + (int64_t)w.h * D, (int64_t)B * S * q_row, flags)) {
#pragma unroll
                    for (int e = 0; e < D / 4; ++e) __stcs(op + e, make_float4(0.f, 0.f, 0.f, 0.f));
                }
                continue;
            }
            float m_run = -INFINITY, l_run = 0.0f;
            const int key_lim = causal ? min(w.p0 + qi + 1, w.n_kv) : w.n_kv;   // keys visible to this row
            for (int j = 0; j < w.nblk; ++j) {
                const int gb = g0 + j;
                ok = mbar_wait(bar.s_full + 8 * (gb % C::NSBUF), (uint32_t)(gb / C::NSBUF) & 1u, abort_flag, flags);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;   // warp-uniform before TMEM access
                tc_fence_after();
                const uint32_t s_col = lane_base + kColS + (uint32_t)((gb % C::NSBUF) * C::S_BUF);
                // S is read out of TMEM twice in 32-column chunks, with the chunk loops rolled: the
                // code stays small (fewer instruction-cache misses) and no more than one chunk of
                // scores is live at a time.
                const int k0 = j * BN;
                const int nvis = min(max(key_lim - k0, 0), BN);     // visible keys of this block
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
                // S holds raw q.k; scores in the exponent's units are s * scale*log2(e) (> 0,
                // so the maximum commutes with the scaling)
                const float m_blk = scale_log2 * fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                // m_use is finite: every row of an item with keys sees at least key 0
                const bool need = m_blk > m_run + kLazyRescale;
                const float m_use = need ? m_blk : m_run;
                const float alpha = need ? fast_exp2(m_run - m_blk) : 1.0f;
                // pass 2: p = 2^(s*c - m); the tensor core truncates f32 operands to TF32, so p is
                // truncated here too and written back over S, and the row sum is taken over exactly
                // those values in eight partial sums (column e into sum e & 7), two columns at a time
                // through the packed f32x2 FMA and add (each lane rounded as the scalar operation;
                // packed sum k holds partial sums 2k and 2k+1).
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
                    // O holds blocks < j once PV_{gb-1} completes; scale it by alpha.  Seeing S_gb
                    // means PV_{gb-NSBUF} completed (issued before QK_gb), so the barrier of
                    // PV_{gb-1}'s buffer is at most one phase behind: the parity wait is exact.
                    ok = mbar_wait(bar.o_done + 8 * ((gb - 1) % C::NSBUF), (uint32_t)((gb - 1) / C::NSBUF) & 1u,
                                   abort_flag, flags);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < C::PV_SPLIT * ((D + 31) / 32); ++c) {
                        if constexpr (D >= 32) {
                            uint32_t wv[32];
                            tmem_ld32(lane_base + kColO + 32 * c, wv);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) wv[e] = __float_as_uint(__uint_as_float(wv[e]) * alpha);
                            tmem_st32(lane_base + kColO + 32 * c, wv);
                        } else {
                            uint32_t wv[16];
                            tmem_ld16(lane_base + kColO + 16 * c, wv);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) wv[e] = __float_as_uint(__uint_as_float(wv[e]) * alpha);
                            tmem_st16(lane_base + kColO + 16 * c, wv);
                        }
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(bar.p_ready + 8 * (gb % C::NSBUF));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            // O / l goes to the item's output staging fills (after its V tiles in the V
            // ring); the V producer stores them to the output by TMA.
            ok = mbar_wait(bar.o_final, (uint32_t)t & 1u, abort_flag, flags);
            if (!(ok = __all_sync(0xffffffffu, ok))) break;
            tc_fence_after();
            // padded rows (and rows without keys) are written as exact zeros, whatever their
            // query held: x * 0 would keep a NaN
            const bool live = qi < w.len && l_run > 0.0f;
            const float inv = live ? 1.0f / l_run : 0.0f;
            const int fs = fv + w.nblk;                          // first staging fill
#pragma unroll 1
            for (int i = 0; ok && i < C::OSLOTS; ++i) {
                ok = mbar_wait(bar.v_loaded + 8 * ((fs + i) % C::NV), (uint32_t)((fs + i) / C::NV) & 1u, abort_flag,
                               flags);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                unsigned char* stage = smem + C::OFF_V + ((fs + i) % C::NV) * C::TILE;
#pragma unroll
                for (int cc = 0; cc < C::OCH; ++cc) {
                    const int c = i * C::OCH + cc;               // column chunk of O
                    unsigned char* dst = stage + cc * (kPfBM * C::CH * 4);
                    if constexpr (C::CH == 32) {
                        uint32_t wv[32];
                        tmem_ld32(lane_base + kColO + 32 * c, wv);
                        if constexpr (C::PV_SPLIT == 2) {            // O = O_a + O_b
                            uint32_t w2[32];
                            tmem_ld32(lane_base + kColO + D + 32 * c, w2);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                wv[e] = __float_as_uint(__uint_as_float(wv[e]) + __uint_as_float(w2[e]));
                        } else {
                            tmem_wait_ld();
                        }
                        if (GUARD && !live) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) wv[e] = 0u;
                        }
                        // 128-byte rows, 16-byte chunk index XOR row bits (the TMA box swizzle)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            *reinterpret_cast<float4*>(dst + r * 128 + (((e & 7) ^ (r & 7)) << 4)) =
                                make_float4(__uint_as_float(wv[4 * e]) * inv, __uint_as_float(wv[4 * e + 1]) * inv,
                                            __uint_as_float(wv[4 * e + 2]) * inv, __uint_as_float(wv[4 * e + 3]) * inv);
                    } else {
                        uint32_t wv[16], w2[16];
                        tmem_ld16(lane_base + kColO, wv);
                        tmem_ld16(lane_base + kColO + D, w2);      // D = 16 always splits PV
                        tmem_wait_ld();
                        if (GUARD && !live) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) wv[e] = w2[e] = 0u;
                        }
                        // 64-byte rows, 64-byte swizzle
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<float4*>(dst + r * 64 + (((e & 3) ^ ((r >> 1) & 3)) << 4)) = make_float4(
                                (__uint_as_float(wv[4 * e]) + __uint_as_float(w2[4 * e])) * inv,
                                (__uint_as_float(wv[4 * e + 1]) + __uint_as_float(w2[4 * e + 1])) * inv,
                                (__uint_as_float(wv[4 * e + 2]) + __uint_as_float(w2[4 * e + 2])) * inv,
                                (__uint_as_float(wv[4 * e + 3]) + __uint_as_float(w2[4 * e + 3])) * inv);
                    }
                }
                fence_proxy_async();                             // generic stores -> TMA reads
                mbar_arrive(bar.v_full + 8 * ((fs + i) % C::NV));
            }
            if (!ok) break;
            fv += w.nblk + C::OSLOTS;
            tc_fence_before();
            mbar_arrive(bar.o_free);     // O may be overwritten by the next item's first PV
            g0 += w.nblk;
            ++t;
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
static inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

template <int D, bool GUARD, bool FILL>
rkv_status launch_prefill_tc_t(const PrefillArgs& a, cudaStream_t stream) {
    using C = PfCfg<D>;
    auto encode = tensor_map_encoder();
    if (!encode) return set_error(RKV_ERR_LAUNCH, "%s: cuTensorMapEncodeTiled unavailable", a.op);
    CUtensorMap tm_k, tm_v, tm_q, tm_o;
    // K/V: interleaved activations [B, S, Hk*D] seen as (Hk*D, S, B), or the cache
    // [B, Hk, max_len, D] seen as (D, max_len, B*Hk)
    const bool cache = a.kv_cache;
    const cuuint64_t dims[3] = {(cuuint64_t)(cache ? D : a.Hk * D), (cuuint64_t)(cache ? a.max_len : a.S),
                                (cuuint64_t)(cache ? (int64_t)a.B * a.Hk : a.B)};
    const cuuint64_t strides[2] = {(cuuint64_t)(cache ? D : a.Hk * D) * 4,
                                   (cuuint64_t)(cache ? a.max_len : a.S) * (cache ? D : a.Hk * D) * 4};
    const PfKv kv = cache ? PfKv{0, a.Hk, 1, a.max_len, a.start_pos} : PfKv{D, 1, 0, a.S, nullptr};
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
        const cuuint32_t qbox[3] = {(cuuint32_t)C::CH, (cuuint32_t)C::BN, 1};   // one query fill
        cr = encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.q), qdims, qstrides, qbox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        // output: same shape as the query; one staged column chunk of a whole tile per store
        // (rows past the sequence end are clipped by the copy engine)
        const cuuint32_t obox[3] = {(cuuint32_t)C::CH, (cuuint32_t)kPfBM, 1};
        if (cr == CUDA_SUCCESS)
            cr = encode(&tm_o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.o, qdims, qstrides, obox, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS) return set_error(RKV_ERR_LAUNCH, "%s: tensor map encode failed (%d)", a.op, (int)cr);
    auto kern = prefill_tc_kernel<D, GUARD, FILL>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return check_launch("prefill: shared-memory attribute");
        attr_done[dev] = true;
    }
    const int n_qtiles = (a.S + kPfBM - 1) / kPfBM;
    const int64_t n_work = (int64_t)n_qtiles * a.B * a.H;
    if (n_work > (int64_t)1 << 30) return set_error(RKV_ERR_UNSUPPORTED, "%s: too many query tiles", a.op);
    // persistent: one CTA per SM (at most one per work item)
    const int sms = sm_count();
    if (sms <= 0) return set_error(RKV_ERR_LAUNCH, "%s: cannot query the SM count", a.op);
    const int grid = (int)(n_work < (int64_t)sms ? n_work : (int64_t)sms);
    kern<<<grid, kPfThreads, C::SMEM, stream>>>(
        tm_k, tm_v, tm_q, tm_o, a.o, a.B, a.S, a.H, a.Hk, a.causal ? 1 : 0, a.seq_lens, a.scale * kPfLog2e, n_qtiles,
        (int)n_work, kv, a.flags);
    if (check_launch(a.op) != RKV_OK) return RKV_ERR_LAUNCH;
    if (FILL) return launch_fill_dependent(a.k, a.v, a.k_cache_out, a.v_cache_out, a.B, a.S, a.Hk, D, a.fill_max_len,
                                           a.flags, stream);
    return RKV_OK;
}

}  // namespace rkv
