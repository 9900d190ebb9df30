"""GB300-native W4A16 group-quantised linear layer.

y = x . dequant(W)^T with x fp16/bf16 [M, K], W 4-bit packed 8 per int32 along
K as [N, K/8], per-group scales [N, K/G] (G in {32, 64, 128}), symmetric
(bias 8) or asymmetric weights (zero points packed 8 per int32 along N as
[N/8, K/G]), fp32 accumulation.

The compute path is the C-ABI shared library ``libw4a16.so`` built from
``csrc/`` (hand-written CUDA for sm_103a); ``binding`` marshals torch tensors
into it.  Nothing here falls back to a CPU or PyTorch implementation: if the
library is missing the calls raise.
"""
from .binding import (  # noqa: F401
    EPI_NONE,
    EPI_SILU_MUL,
    W4A16Error,
    library_path,
    load_library,
    w4a16_clear_device_error,
    w4a16_debug_decode_trace,
    w4a16_debug_set_config,
    w4a16_dequant_debug,
    w4a16_gemm,
    w4a16_dequantize,
    w4a16_gemm_cached,
    w4a16_gemm_chain,
    w4a16_gemm_dense,
    w4a16_gemm_decode_noalloc,
    w4a16_gemm_fused,
    w4a16_gemm_host,
    w4a16_gemm_host_async,
    w4a16_last_device_error,
    w4a16_moe_gemm,
    w4a16_pack,
    w4a16_pack_zeros,
    w4a16_select_path,
)
