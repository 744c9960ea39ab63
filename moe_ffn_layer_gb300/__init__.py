"""MoE FFN layer forward for GB300 (sm_103a): router top-k, counting-sort
permute, tcgen05 grouped GEMMs with fused SiLU*mul, weighted combine, and a
shared expert on a side stream.

The compute path is the C-ABI library ``libmoe_ffn.so`` built from ``csrc/``;
``moe_ffn_layer_gb300.binding`` marshals arguments to it.  Importing this
package loads nothing; the library is loaded on first use and a missing
library is an error, never a fallback.
"""
