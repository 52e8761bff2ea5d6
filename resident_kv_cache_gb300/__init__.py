"""GB300-native resident attention: fused prefill, split-KV batched decode and KV-cache scatter.

The compute path is the C-ABI CUDA library ``librkv_attn.so`` (built for sm_103a from
``csrc/``); ``binding`` marshals arguments to it.  Nothing here computes attention on
the CPU, and every entry point raises if the library is missing.
"""
