"""Paged-KV grouped-query attention for GB300 (sm_103a).

Split-KV decode with an LSE merge and prefix-prefill/extend over a paged KV
cache addressed through per-request block tables, exposed through a C-ABI
library (``include/pa.h``) and the thin ctypes binding in ``binding``.
"""
