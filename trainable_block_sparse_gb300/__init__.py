"""GB300-native VSA (video sparse attention): coarse-to-fine block-sparse attention.

The compute path is the CUDA library libvsa.so (C ABI, include/vsa.h); this
package holds its thin Python binding (`vsa`), the seeded synthetic inputs
(`synth`) and work counts (`flops`).  Importing the package does not load the
library; the first call into `vsa` does, and raises if it is missing.
"""
__all__ = ["synth", "flops", "vsa"]
