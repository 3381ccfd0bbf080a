"""GB300 (sm_103a) block-sparse attention (MSA) hot path.

The compute lives in hand-written CUDA kernels behind a C ABI
(include/msa.h, built into _lib/libmsa_gb300.so); this package is a thin
binding over it.  Importing the package does not need a GPU, but it needs
the built library: there is no CPU fallback.
"""
from .binding import (  # noqa: F401
    ERR_BAD_METADATA, ERR_TMEM_ALLOC, ERR_WAIT_TIMEOUT, EXPORTED, LIB_PATH, MsaError, MsaProblem, Problem,
    attend_decode, attend_decode_noalloc, attend_prefill, check_wait_timeout, error_word, forward,
    index_scores, lib, select_blocks,
)
