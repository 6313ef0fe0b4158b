"""GB300-native paged-KV decode step: KV append, grouped-query paged decode
attention, seeded temperature / top-k / top-p sampling (with min_p,
repetition penalty and log-probs), the frame-local codebook loop, and the
prefill / mixed step (multi-token append, causal paged attention on the
tensor cores), as hand-written CUDA for sm_103a behind a small C ABI
(``include/pkv.h``, ``libpkv.so``).

The Python names below are a thin ctypes binding with the C names minus the
``pkv_`` prefix; they only marshal arguments (torch tensors to device
pointers, the current CUDA stream) -- every step runs in the library's
kernels.  Importing this package does not load the library; the first call
does, and raises if it is missing.
"""

_BINDING = (
    "load", "library_path", "version", "error_string", "PkvError",
    "kv_append", "paged_decode_attn", "decode_workspace_bytes", "paged_decode_attn_static",
    "decode_plan", "paged_decode_attn_planned",
    "kv_append_tokens", "prefill_attn", "prefill_workspace_bytes",
    "seeded_sample", "sample_workspace_bytes", "seeded_sample_ext", "sample_ext_workspace_bytes",
    "codebook_frame_sample", "frame_workspace_bytes",
    "frame_sample", "frame_sample_workspace_bytes",
    "KIND_OTHER", "KIND_AUDIO", "KIND_STOP", "CODE_PAD", "selftest_wait_timeout",
)

__all__ = list(_BINDING)


def __getattr__(name):
    if name in _BINDING:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
