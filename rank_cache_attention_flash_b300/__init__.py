"""LoRA-KV attention for B300 (sm_103a): a C-ABI CUDA library and a thin binding.

The cache of each layer is stored once as a paged base part (K_base, V_base) and
a paged shared-A low-rank part (L_K, L_V); each agent's B_K, B_V are applied at
query time inside the attention kernels.
"""
