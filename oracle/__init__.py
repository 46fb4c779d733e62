"""fp64 CPU oracle for exact attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  See ``oracle/attention.py`` and,
for the FP8 (E4M3) K/V cache, ``oracle/quant.py``.
"""
from .attention import (  # noqa: F401
    attention_backward,
    attention_decode,
    attention_decode_paged,
    attention_forward,
    attention_forward_paged,
    attention_forward_rows,
    cu_from_lengths,
    tile_counts,
    tile_counts_closed_form,
)
