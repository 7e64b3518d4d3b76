"""GB300 (sm_103a) DeepSeek-V4 routed-MoE FFN block with hyper-connections.

The block (``forward_ffn_rows`` of docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs") maps an f32
hyper-connection state [rows, hc, hidden] to a new state: HC prelude (RMSNorm, mix GEMV, sigmoid
pre/post, Sinkhorn comb), ffn_norm, score or hash routing over the experts, grouped routed + shared
SwiGLU experts, weighted reduce, HC post.  It runs in the CUDA kernels of ``libmoe_ffn.so`` behind the
C ABI in ``include/moe_ffn.h``; this package is the Python binding of that ABI (PyTorch supplies
device memory and streams).

Besides the block (``MoeFFN.forward``, ``forward_host``), the handle offers the hyper-connection
prelude and post of a sublayer (``set_attn_hc``, ``hc_pre``, ``hc_post``: the attention sublayer's,
or the FFN's on its own), several layers in one captured submission (``forward_layers``), and
experts in MXFP8 (``set_mxfp8_experts``).
"""
from .api import MoeFFN, MoeFFNError, config_from  # noqa: F401
