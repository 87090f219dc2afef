"""B300-native denoise step of TwoTower block-wise diffusion decoding.

The compute lives in ``libtt_denoise.so`` (CUDA kernels for sm_103a behind the C
ABI of ``include/tt_denoise.h``); ``api`` is its PyTorch binding and ``synth``
draws seeded synthetic inputs.  Build the library with
``python -m block_wise_diffusion_denoise_b300.build``.
"""
from .api import (KVCache, TTError, error_word, tt_block_step, tt_block_step_workspace_size,  # noqa: F401
                  tt_context_block_attn, tt_denoise_attn, tt_denoise_attn_workspace_size, tt_get_device_error,
                  tt_kv_append,
                  tt_unmask, tt_unmask_noalloc, tt_unmask_workspace_size,
                  workspace)
