"""Native Hybrid Attention (NHA) layer operator for NVIDIA GB300 (sm_103a).

The operator ("Native Hybrid Attention for Efficient Sequence Modeling",
Paper-Notes page, section 关键设计/层内混合): m gated linear-RNN key/value
slots fed only by tokens that have left a causal sliding window of w tokens,
the window itself with RoPE, and one 1/sqrt(d) softmax over all m + w keys.
Forward and backward run in the hand-written CUDA kernels of ``libnha.so``
behind the C ABI of ``include/nha.h``; this package is the thin binding.
"""
from ._binding import (  # noqa: F401
    EXPORTS,
    LIB_PATH,
    NHAError,
    launch_count,
    load_library,
    nha_backward,
    nha_backward_varlen,
    nha_decode_prefill,
    nha_decode_state,
    nha_decode_step,
    nha_decode_step_varlen,
    nha_forward,
    nha_forward_noalloc,
    nha_forward_varlen,
    nha_gate_total,
    nha_selftest_wait,
    nha_state_combine,
    nha_varlen_pad,
    nha_varlen_unpad,
    nha_workspace_bytes,
    profile_begin,
    profile_end,
)
