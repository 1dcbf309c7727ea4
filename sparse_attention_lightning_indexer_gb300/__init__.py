"""GB300-native Lightning Indexer (DeepSeek-V4-style sparse attention), sm_103a only.

``ds4idx`` is the Python binding of the C ABI in ``include/ds4idx.h``; ``inputs`` draws the
seeded synthetic workloads; ``build`` compiles the CUDA library in-tree.
"""
