"""GB300-native (sm_103a) EAGLE / EAGLE-2 / EAGLE-3 draft-and-verify cycle.

The compute path is the CUDA library built from csrc/ (libeagle.so, C ABI in
include/eagle.h and include/eagle_ops.h); `api` is a thin ctypes binding over it and
`synth` draws the seeded synthetic weights and prompts. Importing the package does not
load the library; `api.Engine` and the op functions do, and raise if it is not built.
"""
__all__ = ["api", "synth", "build"]
