"""GB300-native speculative tree verify for hybrid Gated DeltaNet + attention
mixer stacks: a C-ABI CUDA library (csrc/) and its thin Python binding."""
