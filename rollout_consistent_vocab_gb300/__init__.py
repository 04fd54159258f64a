"""Strict, batch-invariant token logprob on GB300 (sm_103a).

The compute lives in ``lib/librlk_logp.so`` (CUDA kernels behind a C ABI,
declared in ``include/rlk_logp.h`` and ``include/rlk_norm.h``); this package is its thin Python binding.
"""

from ._binding import (VOCAB_PADDED, VOCAB_REAL, NUM_SHARDS, SHARD_WIDTH, RlkError, LogpArgs,
                       ShardArgs, EXPORTS, load_library, logp_full, logp_pair, logp_restricted,
                       logp_kl, logp_kl_ref, logp_kl_host, logp_kl_host_workspace_bytes, logp_backward, logp_pair_save, logp_backward_saved,
                       logp_autograd, shard_summary,
                       shard_counts, logp_merge, logp_sharded, shard_counts_window,
                       logp_merge_resumable, merge_state, sample, linear_logp, linear_logp_pair,
                       NORM_BINS, norm_bins, sqnorm_accumulate, sqnorm_finalize, reduce_bins_,
                       grad_norm)

__all__ = ["VOCAB_PADDED", "VOCAB_REAL", "NUM_SHARDS", "SHARD_WIDTH", "RlkError", "LogpArgs",
           "ShardArgs",
           "EXPORTS", "load_library", "logp_full", "logp_pair", "logp_restricted", "logp_kl", "logp_kl_ref",
           "logp_kl_host", "logp_kl_host_workspace_bytes",
           "logp_backward", "logp_pair_save", "logp_backward_saved", "logp_autograd", "shard_summary", "shard_counts", "logp_merge", "shard_counts_window", "logp_merge_resumable", "merge_state",
           "logp_sharded", "sample", "linear_logp", "linear_logp_pair", "NORM_BINS", "norm_bins", "sqnorm_accumulate",
           "sqnorm_finalize", "reduce_bins_", "grad_norm"]
