"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench."""
from .workloads import (WORKLOADS, Workload, SparseInputs, MaskedInputs, f32_to_bf16_bits,
                        normal_bf16, uniform_topk, locality_topk, make_indices,
                        make_sparse_inputs, make_masked_inputs, scaled_down)
