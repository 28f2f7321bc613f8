"""Host-streamed, output-tiled linear operator for one GB300 GPU.

``offload_streamed_gb300.tiled_linear`` is the binding of the C ABI
(``include/tiled_linear.h``); ``offload_streamed_gb300.inputs`` draws the
seeded synthetic workloads.  Importing the package loads nothing: the CUDA
library is loaded by the first call into ``tiled_linear``.
"""

__all__ = ["tiled_linear", "inputs"]
