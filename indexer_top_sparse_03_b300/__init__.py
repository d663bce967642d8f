"""B300-native gated sparse attention: indexer -> Top-K -> sparse attention
-> sigmoid output gate, as CUDA kernels for sm_103a behind a C ABI
(include/sparse_attn.h). This package is the thin Python binding over that
library; torch supplies device memory and streams only."""
from .binding import (  # noqa: F401
    ATTN_AUTO, ATTN_TCGEN05, DecodeStep, SA_BF16, SA_F32, SA_FP8_E4M3, SA_OK, SparseAttnError, attention_dense_causal, decode_args,
    decode_workspace_size, device_errors,
    dtype_code, indexer_score, load_library, sparse_attn_decode, sparse_attn_prefill,
    sparse_attn_decode_noalloc, sparse_attn_backward, sparse_attn_prefill_blocks, sparse_attn_prefill_local,
    set_prefill_attention_kernel, status_string,
    topk_select,
)

__version__ = "0.1.0"
