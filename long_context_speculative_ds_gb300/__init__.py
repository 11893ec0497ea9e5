"""GB300 (sm_103a) tree-verify step for long-context speculative decoding.

The compute lives in the C-ABI library built from csrc/ (see include/ds.h);
`binding` is its ctypes binding and `step` allocates the buffers of one
verify step and calls the library.  Importing the package loads nothing.
"""
__all__ = ["binding", "build", "step", "synth"]
