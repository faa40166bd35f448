"""GB300 (sm_103a) page-table-aware fused MoE layer with a shared page pool.

``rimuru`` is the ctypes binding of ``librimuru.so`` (the C ABI in
``include/rimuru.h``); ``device_pool`` places a host image of a pool on the device
through that ABI.  Importing either fails when the library has not been built.
"""
