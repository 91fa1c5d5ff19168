"""fp64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY.  This package is the slow, obviously-correct
definition that the CUDA path is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it.  The product (the C-ABI library and its Python
binding) never imports, links or runs anything in here, and this package
imports nothing from the product.

Every function cites the passage of the source pages it follows:

* "Interrogating the GPU part 5: FlashAttention" (vaibhav016.github.io),
  cited below as [Interrogating-5];
* "FlashAttention versions" (worksonmygpu.com), cited as [FA-versions];
* "FlashAttention" (datarekha.com), cited as [datarekha];
* "LLM Flash Attention" (aicassindra.com), cited as [aicassindra].

Parity status: every function in ``attention`` is pinned by
``tests/test_oracle.py`` (closed forms, invariants, a pure-Python brute
force, finite differences and the worked example that [datarekha] prints),
and every function in ``fp8`` (the FP8 forward's rotation, E4M3 rounding and
block quantisation) by ``tests/test_oracle_fp8.py`` (torch's float8 cast, the
format's codes, closed forms, orthogonality, error bounds and the direction
of the pages' error claim).  No function is "parity unpinned".
"""

from .attention import (  # noqa: F401
    attention_bwd_preprocess_ref,
    attention_bwd_ref,
    attention_fwd_ref,
    attention_probs_ref,
    online_softmax_ref,
    recompute_probs_from_lse_ref,
)
