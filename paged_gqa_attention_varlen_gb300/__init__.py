"""Ragged (varlen) GQA prefill and paged GQA decode for GB300 (sm_103a).

The compute path is the CUDA library libpgqa (C ABI in include/pgqa.h), built with
``paged_gqa_attention_varlen_gb300.build.build()``.  ``api`` is its Python binding;
``workloads`` holds the seeded synthetic input generators.
"""
__all__ = ["api", "build", "workloads"]
