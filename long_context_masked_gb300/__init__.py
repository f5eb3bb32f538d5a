"""GB300-native mask-aware exact softmax attention, forward and backward.

The compute lives in the CUDA library built from ``csrc/`` (C ABI declared in
``include/lca.h``); ``binding`` marshals torch tensors and mask descriptors to
it.  ``inputs`` holds the seeded synthetic workload generators.  Importing the
package loads nothing: the binding and the library are loaded on first use.
"""
_BINDING = ("Plan", "LcaError", "mask_build", "attn_fwd", "attn_bwd", "load_library",
            "library_path", "last_device_error", "selftest_umma", "selftest_wait_timeout",
            "profile_enable", "profile_read", "attn_bwd_noalloc", "block_scores", "block_topk")


def __getattr__(name):
    if name in _BINDING:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
