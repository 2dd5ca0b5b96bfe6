"""DCP causal multi-token MLA verification attention for GB300 (sm_103a).

The computation lives in ``libdcpmla.so`` (hand-written CUDA, C ABI declared in
``include/dcp_mla.h``); this package is its thin Python binding. Importing the
package loads the library and raises if it has not been built: there is no
CPU or PyTorch fallback.
"""

from .binding import (  # noqa: F401
    DCP_OK, DCP_ERR_INVALID_ARG, DCP_ERR_UNSUPPORTED, DCP_ERR_CUDA,
    STATUS_BAD_SEQ_LEN, STATUS_LOCAL_OVER_BOUND, STATUS_BAD_BLOCK_ID, STATUS_BAD_PAGE,
    STATUS_TIMEOUT, STATUS_BAD_SPLIT, KV_BF16, KV_FP8_E4M3, QK_DIM, V_DIM,
    DcpError, Dims, load, library_path,
    dcp_mla_subpage_size, dcp_mla_max_pages, dcp_mla_check_dims, dcp_mla_concurrent_items,
    dcp_mla_metadata, dcp_mla_partial, dcp_mla_partial_hold_q, dcp_mla_partial_packed, dcp_mla_workspace_size, dcp_lse_merge, dcp_last_error, dcp_mla_verify_noalloc,
    dcp_kv_slot_mapping, dcp_kv_write, dcp_a2a_chunk_words, dcp_a2a_pack, dcp_a2a_project,
    dcp_a2a_combine,
)
from .step import (  # noqa: F401
    VerifyStep, choose_num_splits, choose_split_plan, concurrent_items, make_dims, num_sms,
)
from .exchange import A2AExchange, a2a_exchange  # noqa: F401

#: Arithmetic type of the hot path (reported by bench.py): 16-bit tensor-core
#: contractions (f16 for the FP8 cache, bf16 for the BF16 cache), fp32 accumulation,
#: fp32 softmax statistics.
COMPUTE_DTYPE = "f16/bf16 MMA, f32 accumulate"

load()
