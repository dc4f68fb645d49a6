"""Spark-X2.5 gated GQA attention core on one GB300 (sm_103a).

The compute path is the CUDA library libspark_attn.so (C ABI in
include/spark_attn.h); this package only loads it and marshals torch tensors.
"""
from ._binding import (  # noqa: F401
    HEAD_DIM,
    SPARK_DEVERR_POSITION,
    SPARK_DEVERR_TIMEOUT,
    SPARK_GATE_SIGMOID,
    SPARK_GATE_SILU,
    SPARK_LAYER_FULL,
    SPARK_LAYER_SLIDING,
    SPARK_NOALLOC_SCRATCH_BYTES,
    SPARK_OK,
    SparkDeviceFault,
    SparkError,
    as_desc,
    check_device_status,
    layer_desc,
    lib,
    new_workspace,
    spark_attn_decode,
    spark_attn_decode_noalloc,
    spark_attn_decode_workspace_size,
    spark_attn_layer_decode,
    spark_attn_layer_decode_workspace_size,
    spark_attn_layer_prefill,
    spark_attn_layer_prefill_workspace_size,
    spark_attn_prefill,
    spark_attn_prefill_cache,
    spark_attn_prefill_chunk,
    spark_attn_prefill_workspace_size,
    spark_attn_read_status,
    spark_attn_version,
    spark_layer_desc,
    spark_status_str,
)
