"""GB300-native paged-KV attention (decode + extend) behind a C ABI.

The CUDA library (``csrc/``, built into ``_build/libpkv.so``) implements the
calls declared in ``include/pkv.h``; ``binding`` marshals torch tensors into
them. Importing this package does not load the library: the first binding
call does, and raises if it has not been built.
"""
from . import binding  # noqa: F401
from .binding import (PKV_KV_BF16, PKV_KV_FP8_E4M3, PKV_MODE_DECODE, PKV_MODE_DRAFT_EXTEND,  # noqa: F401
                      PKV_MODE_EXTEND, PKV_MODE_IDLE, PKV_MODE_TARGET_VERIFY, PKV_PATH_DECODE, PKV_PATH_EXTEND,
                      PKV_SPEC_DECODE, PKV_SPEC_PREFILL, PagedAttention, PkvError, make_config, pkv_build_metadata,
                      pkv_create, pkv_describe, pkv_destroy, pkv_forward, pkv_forward_decode, pkv_forward_extend,
                      pkv_get_device_error, pkv_get_metadata, pkv_pool_bytes, pkv_select_backend, pkv_set_kv_buffer,
                      pkv_status_string, pkv_workspace_bytes)
