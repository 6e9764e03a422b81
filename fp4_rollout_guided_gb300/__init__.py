"""GB300-native guided-NVFP4 hot path of TRACE (rollout-guided FP4 QAT).

The compute lives in ``libtrace_fp4.so`` (CUDA C++ for sm_103a behind a C
ABI declared in ``include/trace_fp4.h``); :mod:`fp4_rollout_guided_gb300.trace`
is a thin ctypes binding over it, and :mod:`fp4_rollout_guided_gb300.synth`
draws the seeded synthetic workloads.
"""
__all__ = ["synth", "trace"]
