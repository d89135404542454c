"""GB300-native paged KV-cache hot path.

The compute lives in a C-ABI CUDA library (``libpa.so``, built from
``csrc/``); ``pa`` is its thin ctypes binding (argument marshalling only)
and ``workloads`` builds seeded synthetic inputs.  Importing the package
loads nothing; the binding loads the library on first use and raises if it
is missing.
"""
