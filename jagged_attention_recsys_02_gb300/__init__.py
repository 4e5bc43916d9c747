"""GB300 (sm_103a) jagged attention: JFA (softmax) and GDPA (SiLU / GELU).

The compute path is the C-ABI library ``libgdpa.so`` (``include/gdpa.h``);
``binding`` marshals torch tensors into it.  ``workloads`` draws the seeded
synthetic inputs used by the tests and the benchmark.
"""
from . import binding  # noqa: F401
from .binding import gdpa_bwd, gdpa_fwd  # noqa: F401
