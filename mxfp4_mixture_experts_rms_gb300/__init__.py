"""GB300 (sm_103a) MXFP4 routed mixture-of-experts block.

``moe``    ctypes binding of the C-ABI library ``lib/libmoe.so`` (include/moe.h)
``build``  nvcc build of that library
``synth``  seeded synthetic inputs (no block arithmetic)
"""
