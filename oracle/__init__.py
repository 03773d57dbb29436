"""fp64 CPU oracle for the owner-side Muon step (test infrastructure only).

This package is the slow, plain reference that the GPU library is checked
against.  It is TEST INFRASTRUCTURE: only the test-suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product path (``newton_schulz_nesterov_gb300``) never imports, links or
executes anything from here, and nothing here imports the product path.

Everything is computed in float64 with numpy; a dense ``@`` (matmul) is the
only library primitive used as a step.  The algorithm follows the DMuon
documentation pages:

* DMuon "API Reference", section *Optimizer / Muon* (signature defaults
  ``lr=0.02, momentum=0.95, weight_decay=0.0, ns_steps=5, nesterov=True`` and
  the argument note that the Nesterov input is the gradient plus momentum
  times the buffer);
* DMuon "API Reference", section *direct_newton_schulz* (the quintic
  recurrence ``X <- a X + b (X X^T) X + c (X X^T)^2 X``, ``eps=1e-7``);
* DMuon "API Reference", section *gram_newton_schulz_factors* (the
  normaliser is the Frobenius norm plus eps, with the orientation rule that
  works on the transposed matrix when rows > cols);
* DMuon "API Reference", section *YOU_COEFFICIENTS* (the only coefficient
  table the pages print);
* DMuon "HSDP Training", section *What Happens Under the Hood* (the owner
  runs momentum, Newton-Schulz, weight decay and the update).

Pins (tests/test_oracle_pins.py) tie every function here to something other
than itself: the SVD closed form of an odd matrix polynomial, orthogonal
equivariance, transpose symmetry, exact rational arithmetic on 1x1 and
rank-1 cases, and hand-computed momentum/update values.  Two readings are
"parity unpinned" because the pages are silent on them: the update scale
(``scale_mode``) and the coefficient rows used beyond the fifth step.
"""

# oracle.aux_steps holds the fp64 AdamW and segmented-clipping oracle (the
# other parts of Muon.step built here); it is pinned in
# tests/test_oracle_aux_pins.py against hand values and PyTorch's routines.
# oracle.gram holds the Gram-space Newton-Schulz backend with restarts,
# pinned in tests/test_oracle_gram_pins.py to the direct oracle, the SVD
# closed form and the structure of its factors.
# oracle.polar_express derives the Polar Express coefficient table (greedy
# minimax odd quintics with the printed safety factor), pinned in
# tests/test_oracle_polar_express_pins.py by the alternation theorem, its
# chaining and a closed-form limit.
from . import aux_steps  # noqa: F401
from . import gram  # noqa: F401
from . import polar_express  # noqa: F401
from .step import (  # noqa: F401
    YOU_COEFFICIENTS,
    coefficient_rows,
    momentum_update,
    nesterov_input,
    orient,
    frobenius_normalize,
    newton_schulz_direct,
    update_scale,
    apply_update,
    newton_schulz,
    muon_step,
)
