"""Seeded synthetic inputs for the DFlash draft pass.

This package only describes workload shapes and draws random inputs; it holds
none of the method's arithmetic.  Both the CUDA path (through its Python
binding) and the CPU oracle consume exactly the tensors drawn here, so the two
sides always see identical inputs.
"""
from .configs import DraftConfig, Workload, WORKLOADS, get_workload  # noqa: F401
from .generate import (  # noqa: F401
    make_weights, make_features, make_context_lengths, make_page_table,
    make_posterior, make_posterior_with_commit, make_commit_lengths,
    make_anchor, tensor_seed, make_pooled_features, make_match_probs,
)
