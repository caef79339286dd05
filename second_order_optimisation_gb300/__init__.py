"""GB300-native K-FAC curvature step: a C-ABI CUDA library (libkfac_gb300.so)
and a thin ctypes binding (``kfac``)."""
