"""GB300 (sm_103a) hot path of USAF sparse MoE fine-tuning: one MoE layer's train step (routing,
grouped SwiGLU experts forward/backward, gradients at a 0.5% active set, SparseAdam) and the
periodic importance selection and RigL reselection, behind the C ABI in include/usaf.h.

``sparse_moe_fine_gb300.binding`` is the ctypes binding; ``.layer`` a small convenience wrapper
that owns buffers for one layer step; ``.synth`` the seeded synthetic inputs.
"""
