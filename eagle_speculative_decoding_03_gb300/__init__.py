"""GB300-native EAGLE draft-tree expansion step (EAGLE-1 static tree, EAGLE-2
expand-and-rerank dynamic tree, EAGLE-3 fused-feature input).

The compute path is the C-ABI library ``libeagle_draft.so`` built from ``csrc/``
(hand-written CUDA for sm_103a); ``binding`` wraps it with ctypes.  Importing this
package does not load the library: ``binding.load()`` does, and it raises if the
library is missing.
"""
__all__ = ["configs", "synth"]
