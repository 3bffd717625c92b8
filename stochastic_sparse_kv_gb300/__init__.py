"""GB300-native SANTA decode-step attention (stochastic sparse value aggregation).

``santa`` holds the ctypes binding to the CUDA library ``libsanta.so``; ``workloads``
holds the seeded synthetic inputs.  Importing the package loads nothing: the CUDA
library is loaded on first use and its absence raises an error (there is no CPU path).
"""
__all__ = ["santa", "workloads"]
