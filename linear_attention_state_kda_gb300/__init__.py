"""KDA gated delta-rule recurrence on GB300 (sm_103a): a C-ABI CUDA library and its thin
Python binding.

``linear_attention_state_kda_gb300.kda`` holds the binding (one Python function per C entry
point; argument marshalling only). ``inputs`` holds the seeded workload generators. The
binding loads the in-tree ``libkda.so`` on first use and raises if it is missing: there is no
CPU fallback.
"""

__all__ = ["kda", "inputs"]


def __getattr__(name):
    if name in ("kda", "inputs"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
