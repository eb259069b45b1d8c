"""GB300-native fused exact-attention forward (BF16 and FP8 with Hadamard rotation).

The computation lives in libattn46.so (C ABI: include/attn46.h); ``ops`` is
its Python binding and ``synth`` the seeded input generator.  Importing the
package does not load the library; ``ops`` functions load it on first use and
raise if it is missing.
"""

__version__ = "0.1.0"
