"""libsscan: S6 selective-scan forward for NVIDIA B300 (sm_103a), behind a C ABI.

``fwd`` (in ``binding``) marshals torch tensors to the C entry point ``sscan_fwd``; every step of
the scan runs in the library's CUDA kernels. ``inputs`` draws the seeded synthetic workloads.
"""
