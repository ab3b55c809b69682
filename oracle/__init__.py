"""fp64 CPU oracle for DSA sparse-MLA prefill (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does.
"""
from .dsa_oracle import (bf16_to_f64, selected_rows, attend, sparse_prefill, groups, union_pad,
                         union_build, grouped_prefill, topk_to_key_mask, masked_mha_prefill,
                         compare)
