"""GB300-native ZeRO-partitioned mixed-precision Adam shard step.

The compute path is the CUDA library ``libzeroshard.so`` (C ABI declared in
``include/zero_shard.h``); ``binding`` marshals arguments to it.  The library
is loaded on first use and a missing build raises instead of falling back.
"""
__all__ = ["binding", "synth"]
