"""GB300-native submanifold sparse 3D convolution (sm_103a).

The compute path is the C-ABI library ``libvoxelgemm.so`` built from
``csrc/`` (declared in ``include/vg.h``); ``ops`` is its thin Python binding.
Importing this package loads nothing; the first call into ``ops`` loads the
library and raises if it has not been built.
"""
__all__ = ["ops", "synth"]
