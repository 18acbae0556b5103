"""CPU oracle of the activation-sparse FFN decode step (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU legs may import this
package. It shares no code with the CUDA path and imports nothing from it.
"""
from . import sffn_oracle  # noqa: F401
