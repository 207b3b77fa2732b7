"""Plain, slow CPU oracle for the masked attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code with the CUDA path (``block_sparse_attention_masked_gb300``)
and neither side imports the other; both only consume the seeded inputs made
by the ``workloads`` package.

Modules
-------
``dense``  the definition written out in fp64 numpy (row-blocked, every key
           scored, mask applied elementwise afterwards), plus the dense mask,
           the tile enumeration and the exact unmasked-pair count.
``brute``  a pure-Python loop version for N <= 16, written independently from
           the same definitions; it is one of the pins of ``dense``.
``rr_select``  RRAttention's dynamic block selection (round-robin query
           sampling, stride importance, block aggregation, top-tau with the
           last query block kept), in fp64 numpy.
``rr_brute``   the same selection as pure-Python loops for tiny heads, one
           of the pins of ``rr_select``.

Every function of ``dense`` and ``rr_select`` is pinned by a ``-m "not gpu"`` test against
something other than itself (closed forms, the worked example of the SHS
slides, structural special cases, brute force); none is "parity unpinned".
"""

from .dense import (  # noqa: F401
    KINDS,
    allowed,
    inverse_permutation,
    attention,
    attention_probabilities,
    dense_mask_strip,
    received_attention,
    tile_list,
    pair_count,
)
