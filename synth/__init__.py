"""Seeded synthetic inputs for the verify step, shared by the tests and the benchmark.

This module holds none of the verify arithmetic. It only produces logits,
draft tokens and LM-head operands with the shapes and value distributions of
the workloads below; the verify step itself lives in the CUDA library and,
independently, in the oracle.
"""
from .next_rows import NEXT_ROWS, make_contexts, make_draft_lens, make_tree_case
from .workloads import (WORKLOADS, LogitsCase, LMHeadCase, make_logits_case, make_lmhead_case,
                        make_workload, zipf_rank_bias)

__all__ = ["WORKLOADS", "NEXT_ROWS", "LogitsCase", "LMHeadCase", "make_logits_case",
           "make_lmhead_case", "make_workload", "zipf_rank_bias", "make_contexts",
           "make_draft_lens", "make_tree_case"]
