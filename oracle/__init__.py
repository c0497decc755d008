"""CPU oracle for the ternary linear layer — test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import this package. It shares no code with the CUDA path.
"""

from . import ternary_linear  # noqa: F401
