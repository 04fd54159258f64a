"""CPU oracle for the strict token-logprob operator and the deterministic
gradient norm (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product path never does.
"""
from .logp_oracle import (VPAD, VREAL, NSHARD, SHARD_W, InvalidArgument, RowResult,
                          bf16_bits_to_f32, validate, scaled_logits, logp_row,
                          row_logprobs_all, restr_for_support_size, logp_batch,
                          shard_summaries, merge_summaries, top_k_mask, top_p_mask,
                          logp_grad_row, philox4x32_10, philox_uniform_bits, sample_row,
                          SampleResult, linear_logp_row,
                          linear_logp_rows, linear_logp_pair_row, linear_logp_pair_rows)
from .norm_oracle import (NORM_BINS, NAN_BIN, INF_BIN, fp32_squares, sqnorm_bins, bins_exact,
                          finalize as norm_finalize, grad_norm)

__all__ = ["VPAD", "VREAL", "NSHARD", "SHARD_W", "InvalidArgument", "RowResult",
           "bf16_bits_to_f32", "validate", "scaled_logits", "logp_row", "row_logprobs_all",
           "restr_for_support_size", "logp_batch", "shard_summaries", "merge_summaries",
           "top_k_mask", "top_p_mask", "logp_grad_row", "philox4x32_10", "philox_uniform_bits",
           "sample_row", "SampleResult", "linear_logp_row", "linear_logp_rows", "linear_logp_pair_row", "linear_logp_pair_rows",
           "NORM_BINS", "NAN_BIN", "INF_BIN", "fp32_squares", "sqnorm_bins", "bins_exact",
           "norm_finalize", "grad_norm"]
