"""Routed Mixture-of-Experts expert layer for one GB300 (sm_103a).

The compute lives in libmoe.so (C ABI: include/moe.h), built from ``csrc/``
by ``mixture_experts_routed_softmax_gb300.build.build()``. ``layer.MoELayer``
drives the five calls with PyTorch device memory and streams. There is no
CPU path: without the built library every call raises.
"""
