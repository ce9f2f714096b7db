"""Float64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline legs of ``bench.py``; never by the library.
"""
from .attention import (  # noqa: F401
    head_forward, head_probs, head_backward, forward, backward,
    varlen_forward, varlen_backward, decode_forward, decode_partials,
    merge_partials, split_bounds, online_head_forward, gather_pages, paged_decode_forward,
    gqa_forward, gqa_backward, gqa_decode_forward,
)
from .masked import (  # noqa: F401
    window_visible, top_left_causal_visible, block_mask, head_forward_visible, head_backward_visible,
    masked_forward, masked_backward, masked_varlen_forward, masked_varlen_backward,
)
from . import fp8  # noqa: F401  (e4m3 block quantisation with incoherent processing)
from . import paged  # noqa: F401  (write side of the paged cache: append, free list, copy-on-write)
