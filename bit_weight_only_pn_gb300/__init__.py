"""PN weight-only decode GEMV for GB300 (sm_103a).

The CUDA library (``libpn_gb300.so``, C ABI in ``include/pn.h``) is loaded on
first use by :mod:`bit_weight_only_pn_gb300.pn`; importing the package alone
needs no GPU.
"""
__all__ = ["pn", "synth", "build"]
