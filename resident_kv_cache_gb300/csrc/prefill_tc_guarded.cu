// prefill_tc_guarded.cu -- the tensor-core prefill (prefill_tc.cuh) for tiles that may
// reach past a sequence's valid part: per-sequence lengths (attn_prefill with seq_lens)
// and prefill behind an existing cache (attn_prefill_chunked).  Compiled apart from the
// plain variant so the two build in parallel.
//
// Semantics: trustformers-core 0.2.0 src/gpu_ops/cuda/oxicuda/attention.rs,
// fn attention_prefill_gpu_to_gpu (doc: a prefill behind an existing cache runs the
// decode path once per token) and fn attention_decode_gpu_to_gpu.
#include "prefill_tc.cuh"

namespace rkv {

rkv_status launch_prefill_guarded(const PrefillArgs& a, cudaStream_t stream) {
    switch (a.D) {
        case 16: return launch_prefill_tc_t<16, true, false>(a, stream);
        case 32: return launch_prefill_tc_t<32, true, false>(a, stream);
        case 64: return launch_prefill_tc_t<64, true, false>(a, stream);
        case 128: return launch_prefill_tc_t<128, true, false>(a, stream);
    }
    return set_error(RKV_ERR_UNSUPPORTED, "%s: head_dim %d", a.op, a.D);
}

}  // namespace rkv
