"""B300-native selective-scan (S6) forward pass: single direction, Vision Mamba
bidirectional v1/v2 and VMamba SS2D, as hand-written sm_103a CUDA kernels
behind a C ABI (``include/ssm_scan.h``).

The operations are loaded lazily from the compiled library so that
``selective_state_space_111_b300.synth`` (the seeded input generator) can be
imported without it.  Touching any operation when the library is missing
raises immediately: there is no fallback.
"""
_OPS = ("selective_scan_fwd", "bimamba_scan_fwd_v1", "bimamba_scan_fwd_v2",
        "bimamba_scan_fwd_v2_noalloc", "ss2d_scan_fwd", "workspace_bytes", "library_path",
        "SsmError", "version", "set_profile_events", "get_status", "set_cta_channels", "set_prologue_fused",
        "selective_scan_bwd", "bimamba_scan_bwd_v1", "bimamba_scan_bwd_v2", "ss2d_scan_bwd",
        "bwd_workspace_bytes", "bwd_context_bytes", "set_bwd_context", "mamba_prologue_fwd",
        "out_proj_fwd",
        "ss2d_prologue_fwd")


def __getattr__(name):
    if name in _OPS:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)


__all__ = list(_OPS)
