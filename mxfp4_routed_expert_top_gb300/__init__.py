"""GB300 (sm_103a) MXFP4 routed-expert MoE layer: a C-ABI CUDA library
(libdfmoe.so, include/df_moe.h) and its thin Python binding."""
from .binding import (MoE, DfMoeError, Config, LayerWeights, lib, span_bytes_for,  # noqa: F401
                      STACK_RMSNORM_RESIDUAL, PREFILL_MMA_SYNC, MXFP8_ACT, PLANES,
                      SYMBOLS,
                      route_noalloc, Graph, stream_read)
