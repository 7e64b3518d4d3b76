"""GB300 (sm_103a) DeepSeek-V4 routed-MoE FFN block with hyper-connections.

The block (``forward_ffn_rows`` of docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs") maps an f32
hyper-connection state [rows, hc, hidden] to a new state: HC prelude (RMSNorm, mix GEMV, sigmoid
pre/post, Sinkhorn comb), ffn_norm, score or hash routing over the experts, grouped routed + shared
SwiGLU experts, weighted reduce, HC post.  It runs in the CUDA kernels of ``libmoe_ffn.so`` behind the
C ABI in ``include/moe_ffn.h``; this package is the Python binding of that ABI (PyTorch supplies
device memory and streams).
"""
from .api import MoeFFN, MoeFFNError, config_from  # noqa: F401
