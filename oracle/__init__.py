"""fp64 CPU oracle for causal linear attention with the feature map elu(x)+1.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package. The CUDA product path never calls it, and nothing in
here imports the product package: the two share no code.

Every function is the plain mathematical definition from the pages, in float64,
with no blocking, fusion or reordering beyond what that definition states.
"""

from .la_oracle import (  # noqa: F401
    elu,
    phi_elu1,
    phi_elu1_prime,
    phi_identity,
    FEATURE_MAPS,
    forward_masked,
    forward_recurrent,
    decode_step,
    decode_steps,
    output_at,
    backward_recurrent,
    backward_masked,
    loss_dot,
)
from .variants import (  # noqa: F401
    backward_decay,
    decode_steps_decay,
    decode_steps_delta,
    impulse_response,
    half_life,
)
