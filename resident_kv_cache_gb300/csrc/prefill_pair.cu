// prefill_pair.cu -- launches of the CTA-pair prefill (prefill_pair.cuh): head_dim 128 and an
// even number of query heads per kv head, whole sequences (with or without the fused cache
// fill) or tiles that may reach past a sequence (per-sequence lengths, a chunk behind a cache).
//
// Semantics: trueno-gpu 0.4.11 src/memory/resident/attention.rs,
// fn batched_multihead_attention_optimized, and trustformers-core 0.2.0
// src/gpu_ops/cuda/oxicuda/attention.rs, fn attention_prefill_gpu_to_gpu.
#include "prefill_pair.cuh"

namespace rkv {

bool prefill_pair_supported(const PrefillArgs& a) {
    return a.D == PpCfg::D && a.Hk > 0 && a.H % a.Hk == 0 && (a.H / a.Hk) % 2 == 0;
}

template <bool GUARD, bool FILL>
static rkv_status launch_pair_t(const PrefillArgs& a, cudaStream_t stream) {
    using C = PpCfg;
    constexpr int D = C::D;
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
    const cuuint32_t kbox[3] = {(cuuint32_t)C::CH, (cuuint32_t)(C::BN / 2), 1};   // this CTA's 64 keys
    const cuuint32_t vbox[3] = {(cuuint32_t)C::CH, (cuuint32_t)C::BN, 1};         // 128 keys, 32 d
    const cuuint32_t estr[3] = {1, 1, 1};
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    CUresult cr = encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.k), dims, strides, kbox,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr == CUDA_SUCCESS)
        cr = encode(&tm_v, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.v), dims, strides, vbox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr == CUDA_SUCCESS) {
        // query and output [B, S, H*D]: one 32-float column chunk of a 128-row tile per copy
        const cuuint64_t qdims[3] = {(cuuint64_t)a.H * D, (cuuint64_t)a.S, (cuuint64_t)a.B};
        const cuuint64_t qstrides[2] = {(cuuint64_t)a.H * D * 4, (cuuint64_t)a.S * a.H * D * 4};
        const cuuint32_t qbox[3] = {(cuuint32_t)C::CH, (cuuint32_t)kPfBM, 1};
        cr = encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(a.q), qdims, qstrides, qbox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr == CUDA_SUCCESS)
            cr = encode(&tm_o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.o, qdims, qstrides, qbox, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS) return set_error(RKV_ERR_LAUNCH, "%s: tensor map encode failed (%d)", a.op, (int)cr);
    auto kern = prefill_pair_kernel<GUARD, FILL>;
    // per device: the shared-memory attribute, and how many pairs can be resident at once
    static int max_pairs[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return set_error(RKV_ERR_LAUNCH, "%s: device index %d", a.op, dev);
    if (max_pairs[dev] == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return check_launch("prefill: shared-memory attribute");
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * 76, 1, 1);
        cfg.blockDim = dim3(kPfThreads, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0)
            return check_launch("prefill: cluster occupancy");
        max_pairs[dev] = n;
    }
    const int n_qtiles = (a.S + kPfBM - 1) / kPfBM;
    const int64_t n_work = (int64_t)n_qtiles * a.B * a.Hk * (a.H / a.Hk / 2);
    if (n_work > (int64_t)1 << 30) return set_error(RKV_ERR_UNSUPPORTED, "%s: too many query tiles", a.op);
    // persistent: every resident pair walks its share of the items
    const int pairs = (int)(n_work < (int64_t)max_pairs[dev] ? n_work : (int64_t)max_pairs[dev]);
    kern<<<2 * pairs, kPfThreads, C::SMEM, stream>>>(tm_k, tm_v, tm_q, tm_o, a.o, a.B, a.S, a.H, a.Hk,
                                                      a.causal ? 1 : 0, a.seq_lens, a.scale * kPfLog2e, n_qtiles,
                                                      (int)n_work, kv, a.flags);
    if (check_launch(a.op) != RKV_OK) return RKV_ERR_LAUNCH;
    if (FILL) return launch_fill_dependent(a.k, a.v, a.k_cache_out, a.v_cache_out, a.B, a.S, a.Hk, D, a.fill_max_len,
                                           a.flags, stream);
    return RKV_OK;
}

rkv_status launch_prefill_pair(const PrefillArgs& a, bool guard, cudaStream_t stream) {
    if (guard) return launch_pair_t<true, false>(a, stream);
    return a.k_cache_out ? launch_pair_t<false, true>(a, stream) : launch_pair_t<false, false>(a, stream);
}

}  // namespace rkv
