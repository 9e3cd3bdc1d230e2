"""Descriptor-guided masked attention for GB300 (sm_103a).

The compute lives in ``libcm.so`` (C ABI in ``include/cm.h``); ``binding`` is its ctypes
binding, ``specs`` holds the MaskSpecs of the five workloads and ``workloads`` their seeded
synthetic inputs.  Importing the package does not load the library; the first binding call does,
and fails loudly if it has not been built.
"""
