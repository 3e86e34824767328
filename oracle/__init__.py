"""CPU float64 oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import or run anything in this package.  The CUDA path never
calls it, and it shares no code with the CUDA path: the only thing both sides
see is the seeded input data, which the tests pass in as plain arrays.

Modules
-------
attention        the plain definition: materialised S, safe softmax, P V, the
                 log-sum-exp, and the analytic gradients (dQ, dK, dV, D).
online_softmax   an independent restatement of the tiled online-softmax
                 recurrence (running max m, running sum l, rescale alpha), with
                 the "broken" variant that omits the rescale, and the (m, l)
                 merge.  Used only to pin the oracle and the checker.
brute            scalar-loop attention for tiny inputs (no matrix routines).
checker          tolerance comparison with mismatch counting.
fp16_softmax     naive vs max-subtracted softmax rounded to fp16 (overflow pins).
split_kv         attention over key slices and the (m, l, O) merge of the slice
                 results (the split-KV forward).

Parity status: every function here is pinned by tests/test_oracle_*.py against
values printed on the pages (tests/golden/), closed forms, invariants, brute
force and central finite differences.  Bit-exactness against the pages' own
emulator runs is "parity unpinned": their inputs came from a JavaScript RNG
that is not available, so only magnitudes of their printed errors are used.
"""

from .attention import (  # noqa: F401
    forward,
    backward,
    forward_head,
    backward_head,
    probabilities_head,
)
