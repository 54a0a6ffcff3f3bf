"""Seeded synthetic inputs for paged KV append and paged-attention decode.

This package is the one piece of code that both the CUDA path's tests/bench
and the fp64 oracle consume. It holds none of the method's arithmetic: it
draws lengths, block tables, token lists and q/k/v values, and it runs the
host-side block allocator and scheduler that decide which physical blocks a
sequence owns. It never computes a slot, a gather or an attention value.
"""
from .synth import (PagedWorkload, TORCH_DTYPES, chunked_prefill, make_workload, materialize,
                    new_pools, prefill_mha7b, prefill_queries, preset, PRESETS, subset)
from .trace import TraceWorkload, cb_trace, step_inputs, trace_tensors

__all__ = ["PagedWorkload", "TORCH_DTYPES", "make_workload", "materialize", "new_pools",
           "preset", "PRESETS", "TraceWorkload", "cb_trace", "step_inputs", "trace_tensors",
           "chunked_prefill", "prefill_mha7b", "prefill_queries", "subset"]
