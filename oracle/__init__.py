"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library.

Every function follows a passage of the three source pages (cited in each
docstring by page title and section):

* "6.1 FlashAttention V1详解" (AIInfraGuide)             -> cited as [V1详解 §x]
* "A · Flash Attention" (blog.llm.christmas)              -> cited as [A·FA §x]
* "FlashAttention v1～v4" (qscqesze)                      -> cited as [v1～v4 <ver> §x]

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(page values, closed forms, invariants, finite differences, an independent
library routine); none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    to_f64,
    softmax_three_pass,
    online_softmax_blockwise,
    attention_forward,
    attention_forward_rows,
    attention_lse_all_rows,
    attention_abs_weighted_values,
    attention_backward,
    attention_backward_query_rows,
    attention_backward_key_rows,
    flash_forward_kv_outer_v1,
    flash_forward_q_outer,
)
from .fp8 import (  # noqa: F401
    E4M3_MAX,
    e4m3_decode,
    e4m3_encode,
    block_quantize,
    block_dequantize,
    hadamard_rotate_fp32,
    attention_fp8_reference,
)
