"""GB300-native split-KV paged decode attention.

The compute path is the C-ABI CUDA library built from ``csrc/`` (declared in
``include/kf.h``); ``paged_kv_decode_kf_gb300.kf`` is its thin ctypes binding
and ``paged_kv_decode_kf_gb300.workloads`` the seeded input generator. This
package file imports neither, so the input generator can be used on a
machine without a GPU.
"""
__all__ = ["kf", "workloads"]
