"""GB300 resident brute-force top-K retrieval.

The compute path is ``librbf.so`` (hand-written sm_103a CUDA behind the C ABI
in ``include/rbf.h``); this package is its thin Python binding. PyTorch is used
only for device memory and streams.
"""
from ._binding import (  # noqa: F401
    Engine,
    topk_int32_noalloc,
    RbfError,
    load_library,
    lib_path,
    status_string,
    SIGNATURES,
    RBF_OK, RBF_ERR_INVALID_VALUE, RBF_ERR_NOT_READY, RBF_ERR_OUT_OF_MEMORY, RBF_ERR_CUDA,
    RBF_ERR_TIMEOUT, RBF_ERR_UNSUPPORTED, RBF_ERR_BOUNDS, RBF_MAX_K, RBF_MAX_D, RBF_FLAG_FP32_CORPUS,
    RBF_FLAG_BF16_CORPUS, RBF_FLAG_COSINE, RBF_OPT_CTAS_PER_SM, RBF_OPT_STAGE_BYTES, RBF_OPT_SMEM_BUDGET,
    RBF_OPT_TIMEOUT_NS, RBF_OPT_SCHEDULE, RBF_OPT_BATCH_SAMPLE, RBF_OPT_HOST_READ, FAULT_COPY, FAULT_LAUNCH,
)
from ._build import build  # noqa: F401
