"""GB300-native chunked KDA (Kimi Delta Attention): forward and backward for
training on sm_103a, behind a C-ABI library (``libkda.so``, include/kda.h).

``chunk_kda`` / ``recurrent_kda`` live in :mod:`.ops`; the library is loaded on
first use and its absence is an error (there is no fallback path)."""
from .ops import (chunk_kda, chunk_kda_bwd, chunk_kda_bwd_ctx, chunk_kda_bwd_state, chunk_kda_fwd,  # noqa: F401
                  chunk_kda_fwd_ctx, recurrent_kda)
