"""GB300-native forward pass of the gated delta rule (Gated Delta Net recurrence).

The compute path is the C-ABI library ``libgdn.so`` (hand-written CUDA for
sm_103a, sources in ``csrc/``, declarations in ``include/gdn.h``).  The
binding in ``gdn.py`` only marshals tensors into that ABI; importing this
package does not load the library, ``gdn.lib()`` does, and it raises if the
library was not built -- there is no CPU fallback.
"""
from .workloads import WORKLOADS, Workload, generate  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "generate"]
