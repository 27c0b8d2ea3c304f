"""Diagnostics of the kernels, not part of the library's path: the tcgen05 rate benchmark
(tcgen05_rates.cu, a standalone program) and the chunk kernel's stage budget
(chunk_stage_budget.py, through the ``stamps`` build variant)."""
