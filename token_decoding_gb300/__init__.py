"""GB300 (sm_103a) hot path of MARS multi-token generation.

The compute lives in libmars.so (hand-written CUDA, C ABI in include/mars.h);
this package only marshals arguments (``_lib``), builds the library
(``build``) and draws seeded synthetic inputs (``synth``).
"""
from ._lib import (  # noqa: F401
    MARS_DEV_CAPACITY,
    MARS_DEV_LEN_RANGE,
    MARS_DEV_TIMEOUT,
    MarsError,
    accept,
    accept_deferred,
    accept_workspace,
    accept_workspace_size,
    decode_attn,
    decode_attn_deferred,
    lib,
    lm_head_accept,
    lm_head_accept_workspace,
    status_string,
    train_attn,
    train_attn_bwd,
    version,
)
