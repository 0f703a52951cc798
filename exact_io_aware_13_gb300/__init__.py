"""Exact, IO-aware tiled attention on GB300 (sm_103a): forward, backward and the
FlexAttention-style score/mask modifications, as a C-ABI CUDA library with a thin
Python binding."""
from .attention import (MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, MASK_NONE,  # noqa: F401
                        MASK_SLIDING_WINDOW, SCORE_ALIBI, SCORE_DROPOUT, SCORE_NONE, SCORE_SOFTCAP,
                        TILE_EMPTY, TILE_FULL, TILE_PARTIAL, BWD_ALL, BWD_DKDV, BWD_DQ,
                        BWD_ROWDOT, backward, bwd_into, bwd_phases_into,
                        bwd_workspace_size, classify_tiles, device_status, forward, fwd_into,
                        FP8_TILES, FP8_V_TRANSPOSED, fp8_inputs, forward_fp8, fwd_fp8_into,
                        quantize_fp8, decode_paged, decode_paged_into, decode_split_keys,
                        decode_workspace_size, selftest_wait_timeout, check_doc_offsets)
from ._lib import AttnError  # noqa: F401
