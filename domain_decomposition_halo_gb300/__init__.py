"""GB300-native staged-forwarding halo exchange of a 3D domain decomposition.

The compute path lives in libhx (CUDA kernels for sm_103a behind the C ABI of
``include/hx.h``); ``hx`` is its Python binding and ``workloads`` draws the
seeded synthetic inputs.
"""
from .hx import (HX_FLAG_BULK_STORE, HX_FLAG_PDL, HX_FLAG_FINE_WAITS, HX_FLAG_NO_GRAPH, HX_FLAG_RESOLVED,
                 HX_FLAG_SWEEP_FORCES, HX_FLAG_UNORDERED_FORCES, HaloExchange, HXError,
                 load_library, query_plan)

__all__ = ["HaloExchange", "HXError", "load_library", "query_plan", "HX_FLAG_UNORDERED_FORCES",
           "HX_FLAG_NO_GRAPH", "HX_FLAG_FINE_WAITS", "HX_FLAG_SWEEP_FORCES", "HX_FLAG_RESOLVED",
           "HX_FLAG_BULK_STORE", "HX_FLAG_PDL"]
