"""CPU oracle (test infrastructure only).

The oracle is the plain fp64 statement of the denoise step used to check the
CUDA library.  Only tests/, the package smoke check and the benchmark's
CPU-baseline leg may import it; the product path must never depend on it.
"""
from .bd_oracle import (MASK, block_mask, block_attention, current_block_attention,
                        confidence, commit, denoise_step, decode_block,
                        paged_read, append_block, philox4x64_10, uniform01,
                        sample_confidence, denoise_step_sampled, round_bf16, rms_norm,
                        embed, decoder_layer, decoder_forward, truncation_threshold,
                        sample_confidence_truncated, silu, mlp_residual)

__all__ = ["MASK", "block_mask", "block_attention", "current_block_attention",
           "confidence", "commit", "denoise_step", "decode_block",
           "paged_read", "append_block", "philox4x64_10", "uniform01",
           "sample_confidence", "denoise_step_sampled", "round_bf16", "rms_norm",
           "embed", "decoder_layer", "decoder_forward", "truncation_threshold",
           "sample_confidence_truncated", "silu", "mlp_residual"]
