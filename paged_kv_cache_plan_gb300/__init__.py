"""Paged-KV split-KV decode attention for GB300 (sm_103a).

The product is the C-ABI library libpkvd.so (include/pkvd.h): a host split
planner plus hand-written CUDA kernels (stage-1 split attention, stage-2
log-sum-exp merge). This package holds its sources (csrc/), its build
script, the ctypes binding with the same entry-point names, and the seeded
synthetic workload generator. Importing the package does not load the CUDA
library; the first call does, and fails loudly if it is not built.
"""
from .api import (Plan, cp_decode, cp_ranges, decode_merge_ranks, decode_plan,
                  decode_plan_compute, decode_plan_cp, decode_plan_cp_compute, decode_plan_ex,
                  decode_plan_prefix, decode_plan_prefix_compute, decode_run, decode_run_timed,
                  gather_ranks, make_desc, plan_for_case, prefill_d64, run_case,
                  selftest_wait_timeout)

__all__ = ["Plan", "decode_plan", "decode_plan_ex", "decode_plan_prefix", "decode_run",
           "decode_run_timed", "decode_plan_compute", "decode_plan_prefix_compute", "make_desc",
           "plan_for_case", "prefill_d64", "run_case", "selftest_wait_timeout", "cp_ranges",
           "decode_plan_cp", "decode_plan_cp_compute", "decode_merge_ranks", "gather_ranks",
           "cp_decode"]
