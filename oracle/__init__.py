"""Plain CPU oracle for the routed-MoE FFN block.

TEST INFRASTRUCTURE ONLY.  Imported by tests/, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline/reference leg, never by the library.  See ``moe_ffn.py``.
"""
from .moe_ffn import *  # noqa: F401,F403
from .moe_ffn import forward_ffn_rows, hc_sublayer_pre, prelude_and_route  # noqa: F401
