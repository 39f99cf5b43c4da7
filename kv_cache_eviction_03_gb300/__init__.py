"""H2O heavy-hitter KV-cache eviction: GB300 (sm_103a) decode and prefill.

The compute path is the C-ABI library built from `csrc/` (see
`include/h2o.h`); `binding` is its thin ctypes wrapper.  Importing this
package does not load the library; `binding.lib()` does, and raises if it is
missing.
"""
__all__ = ["binding", "workload", "accounting"]
