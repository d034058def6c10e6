"""Paged KV attention for GB300 (sm_103a).

Exact softmax attention over a paged KV cache of 16-token blocks for a
flattened, variable-length serving batch, plus the slot-mapped KV write.  The
compute runs in hand-written CUDA kernels behind the C ABI of
``include/pkv.h`` (``_lib/libpkv.so``); this package is its Python binding
(``pkv_write``, ``pkv_attention_varlen``, their 8-bit E4M3-cache forms
``pkv_write_e4m3`` and ``pkv_attention_varlen_e4m3``, the shared-prefix
``pkv_cascade_attention``, ``pkv_num_splits``,
``pkv_workspace_bytes``, ``pkv_status_string``) and the runner-side metadata
builder (``metadata.build``), and a decode runner that replays steps from a
ladder of captured CUDA graphs (``graphs.DecodeGraphRunner``).  PyTorch supplies
device memory, streams and graph capture.
"""

from . import graphs, metadata  # noqa: F401
from ._binding import (EXPORTS, FLAG_BAD_BLOCK, FLAG_BAD_LENGTHS, FLAG_BAD_SLOT,  # noqa: F401
                       FLAG_TIMEOUT, PKV_DECODE_MAX_QLEN, PkvError, lib, pkv_attention_varlen,
                       pkv_attention_varlen_e4m3, pkv_attention_varlen_noalloc,
                       pkv_build_metadata,
                       pkv_cascade_attention, pkv_cascade_splits, pkv_cascade_workspace_bytes,
                       pkv_num_splits, pkv_stage_inputs, pkv_status_string, pkv_workspace_bytes,
                       pkv_write,
                       pkv_write_attention_varlen, pkv_write_attention_varlen_e4m3,
                       pkv_write_e4m3)
