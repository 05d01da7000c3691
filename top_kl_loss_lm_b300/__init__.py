"""Fused top-K KL distillation head for B300 (sm_103a).

The compute runs in ``libkdtopk.so`` (CUDA kernels behind a C ABI declared in
``include/kd_topk_kl.h``); ``binding`` marshals torch tensors into those calls.
Importing the package does not load the library; the first call does, and it
raises if the library is missing.
"""
