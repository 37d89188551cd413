"""GB300-native hot path of DWDP (Distributed Weight Data Parallelism).

The compute lives in ``libdwdp.so`` (hand-written CUDA for sm_103a behind a C
ABI, declared in ``include/dwdp.h``); ``binding`` marshals arguments to it.
``inputs`` generates seeded synthetic layers.
"""
