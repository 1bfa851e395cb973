"""GB300 (sm_103a) quantized MoE decode layer: Python binding of the C ABI.

The layer's arithmetic runs in the CUDA library ``libmoe_gb300.so`` (built by
``quantized_moe_decode_gemv_gb300.build.build()``); this package only marshals
arguments.  Importing a name that needs the library raises if it is missing.
"""
from ._capi import (  # noqa: F401
    MoEConfig, MoEError, MoELayer, load_library, moe_layer_create, moe_layer_destroy,
    moe_layer_device_status, moe_layer_forward, moe_layer_forward_ex, moe_layer_forward_host,
    moe_layer_set_path, moe_layer_validate, moe_router_topk_noalloc, torch_act_dtype, upload_arrays, SIGNATURES, LIB_PATH,
)
