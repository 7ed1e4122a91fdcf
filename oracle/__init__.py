"""CPU oracle for the nanochat pretraining step (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg may import
this package. It shares no code with the CUDA library and the library never
calls it: there is no CPU fallback anywhere in the product path.
"""

from .model import (EPS, HEAD_DIM, IGNORE, ROPE_BASE, Shape, backward, causal_attention,
                    causal_attention_backward, cross_entropy_backward,
                    cross_entropy_rows, forward, layout, param_count, relu2,
                    relu2_backward, rmsnorm, rmsnorm_backward, rope,
                    rope_angles, rope_backward, split_packed, step, step_accumulated, unpack)
from . import infer, optim
