"""GB300 layer-boundary library: fold K partial sums (or a deferred MoE finalize)
into the residual stream and produce the consumer's RMSNorm / FP8 input in one pass.

The compute path is the C-ABI library ``liblb.so`` (hand-written sm_103a kernels);
``layer_boundary_fusion_gb300.lb`` is its thin ctypes binding.  Importing this
package loads nothing; the binding loads the library on first use and raises if it
is missing.
"""
__all__ = ["workloads"]
