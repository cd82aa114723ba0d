"""GB300-native XPress Jacobi draft pass (speculative decoding).

The compute path is the C-ABI library ``libxpress.so`` built from the CUDA
sources in ``csrc/`` for sm_103a; ``xpress`` is its thin Python binding
(argument marshalling only).  ``synth`` draws the seeded synthetic inputs.
Importing the package loads nothing; ``xpress.lib()`` loads the library and
raises if it is missing.
"""

__all__ = ["xpress", "synth"]
