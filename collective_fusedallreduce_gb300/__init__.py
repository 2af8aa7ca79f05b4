"""GB300-native fused and decomposed collectives over N logical ranks in one GPU.

The compute path is the C-ABI library ``libcoco.so`` (hand-written sm_103a
kernels); ``coco`` is its thin Python binding. Nothing here computes on the
CPU: if the library is missing, importing the binding raises.
"""
