"""GB300 (sm_103a) fused 8-bit blockwise AdamW with stochastic rounding.

The compute lives in libq8adamw.so (C ABI: include/q8adamw.h); this package
is its Python binding (same names as the C entry points) plus a torch.optim
front end (bit_blockwise_adamw_gb300.optim).
"""
from ._binding import (  # noqa: F401
    BLOCK, EXPORTS, MAX_STEP, SIGNED, SMALL_NUMEL, UNSIGNED, HParams, LionHParams, MomentumHParams,
    Q8Error, Tensor8, Tensor16, adamw8bit_sr_step, adamw_bf16_sr_step, hparams, library_path,
    lion8bit_sr_step, lion_hparams, load_library, momentum8bit_sr_step, momentum_hparams,
    pack_tensor8, pack_tensor16, q8_abi_version, q8_blockwise_dequantize, q8_blockwise_quantize,
    q8_codebook_init, q8_last_error, q8_philox_fill, q8_prepare_device, q8_selftest_sqrt_div)
