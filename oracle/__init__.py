"""CPU float64 oracle for causal prefill attention (test infrastructure only).

This package is the independent checker of the CUDA path. Only the test suite,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may import it. The product path never calls it, and it shares
no code, tables or helpers with the CUDA library.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle.py`` (closed forms, invariants, brute force, a library
routine for the special case, a hand-worked example and the e4m3 format facts
that the ZYFA README prints).
"""

from .attention import (  # noqa: F401
    attention_f64,
    attention_rows_f64,
    causal_probs_f64,
    decode_inputs_f64,
)
from .formats import bf16_to_f64, e4m3_to_f64  # noqa: F401
from .rotation import (  # noqa: F401
    dct3_f64,
    fp8_quantize_rotated_f64,
    hadamard_f64,
    rotate_f64,
    rotation_f64,
)
