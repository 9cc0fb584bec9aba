"""GB300-native weight-absorbed MLA decode.

The compute path is the C-ABI library built from ``csrc/`` (declared in
``include/mla.h``); ``mla`` is its thin ctypes binding and ``workloads`` draws the
seeded synthetic inputs.  Importing the package loads nothing: the library is
opened on first use, and every call fails loudly if it is missing.
"""
