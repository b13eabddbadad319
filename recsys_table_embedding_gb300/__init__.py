"""GB300-native table-batched embedding (TBE) training hot path.

The compute lives in libtbe_gb300.so (hand-written CUDA for sm_103a behind
the C ABI in include/tbe.h); ``tbe`` is its ctypes binding.
"""
from .tbe import (TBE, Batch, Meta, Tables, TbeError, config, lib, meta_view, tbe_backward_rowwise_adagrad,
                  tbe_forward, tbe_meta_bind, tbe_preprocess, tbe_preprocess_static, tbe_query_sizes,
                  tbe_select_path)

__all__ = ["TBE", "Batch", "Meta", "Tables", "TbeError", "config", "lib", "meta_view",
           "tbe_backward_rowwise_adagrad", "tbe_forward", "tbe_meta_bind", "tbe_preprocess",
           "tbe_preprocess_static",
           "tbe_query_sizes", "tbe_select_path"]
