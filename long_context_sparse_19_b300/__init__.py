"""B300-native compressed-sparse-attention (CSA / HCA) hot path.

The computation lives in ``libcsa.so`` (hand-written sm_103a CUDA kernels behind the C ABI of
``include/csa.h``); this package is its thin Python binding. Importing it loads the library and
fails loudly if it has not been built.
"""
from .binding import (  # noqa: F401
    CSA_BF16, CSA_ERR_DEVICE, CSA_ERR_DEVICE_TIMEOUT, CSA_F32, CSA_FP4, CSA_FLAG_SIMT, EXPORTS, Cache, Config, CsaCache,
    CsaConfig, CsaError, cache_tensor, csa_cache_bytes, csa_compress, csa_decode, csa_get_device_status, csa_index_topk, csa_index_topk_static,
    csa_prefill, csa_sparse_attn, csa_sync_status, csa_index_topk_shard, csa_topk_merge, csa_sparse_attn_shard,
    csa_attn_merge,
    csa_status_string, csa_workspace_bytes, load, workspace, csa_launch_count, csa_profile_begin,
    csa_profile_end, STAGES,
)

load()
