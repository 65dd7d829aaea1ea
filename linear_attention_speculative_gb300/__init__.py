"""Fused causal-conv1d + Kimi Delta Attention multi-token-prediction verify
decode for GB300 (sm_103a).

    from linear_attention_speculative_gb300 import kda
    kda.conv_verify(mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0,
                    "softplus", o, inter_ssm, conv_snapshots, workspace)

`kda` is the ctypes binding of the C ABI (include/kda_verify.h); `workloads`
draws seeded synthetic inputs.  Submodules are imported on demand so that the
input generator can be used without the CUDA library.
"""

__all__ = ["kda", "workloads"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
