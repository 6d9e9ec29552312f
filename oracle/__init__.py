"""Test infrastructure only: the fp64 CPU oracle for rank-compressed paged attention."""
from .rcp_oracle import (append_kv, attend, decode_attn, gather_request,  # noqa: F401
                         prefill_attn)
