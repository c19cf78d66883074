"""GB300-native block-sparse attention backward (and its companion forward).

The compute path is the C-ABI library ``libbsa.so`` (header ``include/bsa.h``),
built from the CUDA sources under ``csrc/`` for sm_103a. This package only
marshals arguments into that library; importing it never loads CUDA, and every
compute call raises if the library has not been built.
"""
from .binding import (bsa_grad_workspace_size, bsa_grad, bsa_fwd_workspace_size,  # noqa: F401
                      bsa_fwd, bsa_mask_compact, bsa_mask_compact_noalloc, bsa_check_status,
                      check_pending_status,
                      BsaError,
                      block_sparse_attention_grad, block_sparse_attention_fwd,
                      block_sparse_attention, BlockSparseAttentionFunction,
                      load_library, library_path, NO_WINDOW)
