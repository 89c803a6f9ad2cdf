"""Float64 CPU oracle for exact tiled attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import, call or execute anything
in this package.  The product path (the CUDA library under
``exact_tiled_attention_11_gb300`` and its Python binding) never imports it,
and this package imports nothing from the product: the two share no code.
Only the seeded input generators (``exact_tiled_attention_11_gb300.workloads``,
which hold none of the attention arithmetic) feed both sides.

Everything is plain NumPy in float64, one (batch, head) at a time, written so
that it can be checked against the pages by eye:

* ``attention``        -- the plain definition (materialised S, stable softmax,
                          P.V, log-sum-exp), which exact tiled attention reaches
                          up to rounding order; ``attention_weights`` returns
                          the softmax weights P of selected rows (the error
                          bound of FP8 attention weighs each key's rounding by
                          them).
* ``tiled_attention``  -- the block-wise algorithm itself (online softmax over
                          K/V tiles, causal tile skipping), reporting the block
                          pairs it visited.
* ``partial_state`` / ``merge_partials`` / ``finalize`` -- the (m, l, o~)
                          partial results over a key subset and their exact
                          merge rule.
* ``decode_paged``     -- one query token per sequence against a paged, ragged
                          KV cache gathered through a page table.
* ``cascade_decode``, ``varlen_attention``, ``paged_prefill`` -- a shared prefix
                          plus own suffix; ragged (indptr) batches; ragged
                          query chunks against a paged cache.
* ``fp8`` (submodule)  -- FP8 attention's inputs: the random orthogonal
                          (Hadamard) transform of Q and K, block quantisation to
                          e4m3 with one scale per 128-row block, and the exact
                          attention of the dequantised blocks.

Pins (``tests/test_oracle_pins.py``, ``-m "not gpu"``): the worked examples the
pages print, a scalar pure-Python brute force on tiny inputs, closed forms
(K = 0, one key), invariants (block-shape independence, partition/merge
independence, convex combination, no overflow at large scores) and the causal
block-pair counts the pages report; ``tests/test_oracle_fp8.py`` pins the FP8
part against PyTorch's e4m3 conversion, scipy's Hadamard matrix, orthogonality,
a scalar brute force and the quantisation error bound.  No function here is
unpinned.
"""
from .attention import (  # noqa: F401
    attention,
    attention_rows,
    attention_weights,
    tiled_attention,
    partial_state,
    merge_partials,
    finalize,
    decode_paged,
    cascade_decode,
    varlen_attention,
    paged_prefill,
    gather_sequence,
    to_f64,
)
from . import fp8  # noqa: F401
