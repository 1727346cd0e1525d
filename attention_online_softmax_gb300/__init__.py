"""GB300-native fused attention: softmax as a monoid over key blocks.

Prefill (``attn_fwd``) and paged split-KV decode (``attn_decode_paged``) run in
hand-written sm_103a CUDA kernels behind the C ABI declared in
``include/attn.h``.  ``attention_online_softmax_gb300.abi`` is the thin ctypes
binding with the same names; importing it loads the compiled library and fails
loudly when it is missing.  ``inputs``, ``configs`` and ``roofline`` are plain
Python helpers (seeded synthetic inputs, workload table, work/traffic
counters) and do not touch the library.
"""

__all__ = ["abi", "inputs", "configs", "roofline"]
