"""GB300 (sm_103a) hot path of block speculative verification.

The compute lives in a C-ABI CUDA library (``csrc/``, declared in
``include/vq.h``); ``binding`` marshals torch tensors into it. Importing this
package does not load the library: ``binding.lib()`` does, and fails loudly
when it has not been built.
"""
