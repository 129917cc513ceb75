"""GB300-native Kimi Delta Attention (KDA) gated delta-rule recurrence.

The compute lives in the C-ABI library ``libkda.so`` (hand-written CUDA for
sm_103a, declared in ``include/kda.h``). ``kda`` is its thin ctypes binding;
``synth`` draws the seeded synthetic inputs. Importing the package loads
nothing: the library is opened on the first call and an error is raised if
it has not been built.
"""
__all__ = ["kda", "synth"]
