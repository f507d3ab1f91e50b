"""GB300-native DeepSeek Sparse Attention (DSA) decode path.

The compute lives in ``libdsa.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/dsa.h``); ``api`` is a thin ctypes binding over it.
Importing the package does not load the library: the first call into ``api``
does, and fails loudly if it has not been built.
"""
