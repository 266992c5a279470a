"""B300-native (sm_103a) DeepSeek-V4 hybrid attention: CSA + HCA + SWA.

The compute lives in the CUDA library `libhattn.so` behind the C ABI declared
in include/hattn.h; `hattn` is its thin ctypes binding.
"""
__all__ = ["hattn", "synth"]
