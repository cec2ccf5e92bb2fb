"""GB300-native KPool DSA indexer selection.

The compute path is the CUDA library built from ``csrc/`` (C ABI declared in
``include/kpool.h``); :mod:`.kpool` is its thin ctypes binding and
:mod:`.workloads` holds the seeded synthetic inputs. Importing the package
loads nothing: the library is opened on the first call into the binding.
"""

__all__ = ["kpool", "workloads"]
__version__ = "0.1.0"
