"""GB300-native FlashMap one-jump block-draft step.

The compute path is the C-ABI library built from ``csrc/`` (see
``include/flashmap.h``); ``_lib`` is its thin ctypes binding. ``synthetic`` draws
seeded inputs for tests and benchmarks.
"""
