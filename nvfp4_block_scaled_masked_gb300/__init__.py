"""Masked, block-scaled NVFP4 grouped GEMM-NT for GB300 (sm_103a).

``binding`` wraps the C-ABI library ``libnvfp4gg.so`` (hand-written CUDA
kernels); ``workloads`` draws seeded synthetic inputs.  Importing the package
loads nothing: the library is opened on first use of ``binding``.
"""
