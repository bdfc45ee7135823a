"""Batch-1 autoregressive decode engine for one GB300 (sm_103a).

The engine is the CUDA library libkie.so (C ABI in include/kie.h); this package
only builds and binds it.  See ``kie.Engine``.
"""
from .kie import (Engine, KieError, convert_fp8_e5m2, load, make_config, quantize_int4_g128,  # noqa: F401
                  quantize_kv_u8)
