"""EasySpec layer-parallel speculative decoding on one B300 (sm_103a).

The compute path is the C-ABI library ``libeasyspec.so`` (hand-written CUDA);
``layer_drafting_draft_b300.easyspec`` is its thin ctypes binding.  Importing
this package loads nothing: the library is opened on first use, and a missing
library is an error, never a fallback.
"""
