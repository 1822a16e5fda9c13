"""B300-native (sm_103a) forward pass of a sparse Mixture-of-Experts FFN layer.

The compute path is the C-ABI library ``libmoe.so`` built from ``csrc/``;
``binding`` marshals arguments to it with ctypes.  ``workloads`` and
``synth`` describe and draw the layer shapes.  The library is loaded on first
use, so importing this package needs no GPU.
"""

from .workloads import WORKLOADS, Workload  # noqa: F401
