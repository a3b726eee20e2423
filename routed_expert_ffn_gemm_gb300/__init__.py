"""GB300-native forward of one Mixture-of-Experts FFN layer.

The compute path is a C-ABI CUDA library (``libmoe_gb300.so``, kernels for
sm_103a) reached through the thin ctypes binding in ``api``.  Importing this
package does not load the library; the first call into ``api`` does, and
fails loudly if it has not been built.
"""

from .inputs import MoEShape, WORKLOADS, DECODE_T  # noqa: F401

__all__ = ["MoEShape", "WORKLOADS", "DECODE_T"]
