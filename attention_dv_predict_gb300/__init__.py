"""Contextually sparse (DejaVu) single-layer decode for GB300 (sm_103a).

``attention_dv_predict_gb300.dv`` is the Python binding of the C-ABI library
``libdv.so`` (argument marshalling only; every step runs in the library's CUDA
kernels).  Importing it fails loudly if the library has not been built.
``attention_dv_predict_gb300.traffic`` is the byte model used for rooflines.
"""

__all__ = ["dv", "traffic"]
