// prefill_tc.cu -- launches of the tensor-core prefill (prefill_tc.cuh) for whole
// sequences of interleaved activations (with or without the fused cache fill), and the
// dispatch between the variants.
//
// Semantics: trueno-gpu 0.4.11 src/memory/resident/attention.rs,
// fn batched_multihead_attention_optimized, and trustformers-core 0.2.0
// src/gpu_ops/cuda/oxicuda/attention.rs, fn attention_prefill_gpu_to_gpu.
#include "prefill_tc.cuh"

namespace rkv {

rkv_status launch_prefill_guarded(const PrefillArgs& a, cudaStream_t stream);   // prefill_tc_guarded.cu

rkv_status launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    // per-sequence lengths or keys from the cache: tiles may reach past a sequence
    const bool guard = a.kv_cache || a.seq_lens;
    // head_dim 128 with pairs of query heads per kv head: two CTAs share each product
    if (prefill_pair_supported(a)) return launch_prefill_pair(a, guard, stream);
    if (guard) return launch_prefill_guarded(a, stream);
    if (a.k_cache_out) {                // whole sequences, their K/V also written to the cache
        switch (a.D) {
            case 16: return launch_prefill_tc_t<16, false, true>(a, stream);
            case 32: return launch_prefill_tc_t<32, false, true>(a, stream);
            case 64: return launch_prefill_tc_t<64, false, true>(a, stream);
            case 128: return launch_prefill_tc_t<128, false, true>(a, stream);
        }
    } else {
        switch (a.D) {
            case 16: return launch_prefill_tc_t<16, false, false>(a, stream);
            case 32: return launch_prefill_tc_t<32, false, false>(a, stream);
            case 64: return launch_prefill_tc_t<64, false, false>(a, stream);
            case 128: return launch_prefill_tc_t<128, false, false>(a, stream);
        }
    }
    return set_error(RKV_ERR_UNSUPPORTED, "%s: head_dim %d", a.op, a.D);
}

}  // namespace rkv
