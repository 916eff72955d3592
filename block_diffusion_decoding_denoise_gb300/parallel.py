"""One sequence's denoise step split across GPUs.

The path shards by sequence with no exchange (bench.py runs replicas).  Two
splits inside a sequence need one exchange each, and the library provides the
two sides of it (see bd.h):
  vocabulary-parallel LM head: every rank reduces its slice of W to one
    12-byte state per position (bd_confidence_shard); the states are gathered
    and merged into p_max and argmax before the commit (bd_commit_shards);
  KV-split attention: every rank's (m, l, O) partials per query row are
    gathered and merged (bd_merge_attention_partials).
The exchange itself is the caller's collective (torch.distributed here, NCCL
on GPUs); the host merges serve ranks that gather on the CPU.
"""
from __future__ import annotations

import numpy as np
import torch

from . import bd

RECORD = np.dtype([("m", "<f4"), ("s", "<f4"), ("idx", "<i4")])


def vocab_shard_bounds(vocab: int, world: int, rank: int) -> tuple[int, int]:
    """[start, end) of rank's vocabulary slice: contiguous, sizes differ by at most one."""
    base, extra = divmod(vocab, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def vocab_parallel_commit(h, w_shard, vocab_offset, vocab, threshold, tokens, p_max, argmax,
                          n_committed, n_masked, ws, group=None, dev_status=None):
    """One greedy confidence/commit call with W split over the ranks of
    `group`: each rank holds rows [vocab_offset, vocab_offset + len(w_shard))
    of W and the same h and tokens.  One all-gather of 12 bytes per position;
    every rank then applies the same commit."""
    import torch.distributed as dist
    B, L, _ = h.shape
    records = torch.empty(B * L, bd.RECORD_INTS, dtype=torch.int32, device=h.device)
    bd.bd_confidence_shard(h, w_shard, vocab_offset, tokens, records, ws, dev_status)
    world = dist.get_world_size(group)
    gathered = torch.empty(world, B * L, bd.RECORD_INTS, dtype=torch.int32, device=h.device)
    dist.all_gather_into_tensor(gathered, records, group=group)
    bd.bd_commit_shards(gathered, vocab, threshold, tokens, p_max, argmax, n_committed,
                        n_masked, dev_status)


def merge_records_host(gathered: np.ndarray) -> np.ndarray:
    """Merge records gathered on the host: [num_shards, n] RECORD -> [n]."""
    return bd.bd_merge_conf_records_host(np.ascontiguousarray(gathered, dtype=RECORD))


def merge_attention_host(m: np.ndarray, l: np.ndarray, o: np.ndarray) -> np.ndarray:
    """Merge KV-split partials gathered on the host (float32):
    m, l [num_shards, rows], o [num_shards, rows, D] -> [rows, D]."""
    return bd.bd_merge_attention_partials_host(m, l, o)
