"""Row-sharded search across ranks (one GPU each): partition, exchange, merge.

A corpus too large for one GPU is split into contiguous row shards, one per
rank (GPU-Resident Top-K for Agentic RAG, section 4 step 1 on where the corpus
lives, and section 9, which names sharding across GPUs as the way past one
GPU's memory). Each rank runs the unchanged single-GPU search on its shard,
with the shard's first global row as the engine's index offset
(upload_corpus_shard), so its K best come out with global row indices and
global tie order. One exchange per query batch (an all-gather of 2 K words per
query and rank) gives every rank all G lists, and the library's merge kernel
(merge_shard_topk_dev) combines them under the same ordering rule: the result
is the one a single GPU holding the whole corpus returns.

This module is host logic only: the partition, the exchange through
torch.distributed (NCCL with device tensors, gloo with CPU tensors) and the
order of the calls. Every score and every comparison runs in the library's
kernels.
"""
from __future__ import annotations


def shard_rows(n_total: int, world: int, rank: int) -> tuple[int, int]:
    """(first global row, rows) of rank's shard: contiguous ranges in rank
    order, the first n_total % world shards one row longer."""
    if world < 1 or not 0 <= rank < world or n_total < world:
        raise ValueError("need 0 <= rank < world <= n_total")
    base, extra = divmod(n_total, world)
    row0 = rank * base + min(rank, extra)
    return row0, base + (1 if rank < extra else 0)


def exchange(idx, score, group=None):
    """All-gather every rank's best-first lists: idx (int32) and score (fp32)
    of one shape [b, k] (or [k]) on each rank become [g, b, k] (or [g, k]),
    rank r's lists at [r] -- the layout merge_shard_topk_dev reads. One
    collective of the packed pair; device tensors under NCCL, CPU tensors
    under gloo."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    packed = torch.stack([idx.contiguous(), score.contiguous().view(torch.int32)])
    parts = [torch.empty_like(packed) for _ in range(world)]
    dist.all_gather(parts, packed, group=group)
    out = torch.stack(parts)  # [g, 2, ...]
    return out[:, 0].contiguous(), out[:, 1].contiguous().view(torch.float32)


class ShardedSearch:
    """This rank's part of a row-sharded search: an engine over its shard, the
    exchange, and the merge. Collective: every rank calls every method with
    the same arguments (queries, K) in the same order."""

    def __init__(self, rbf, n_total: int, d: int, max_k: int, world: int, rank: int, group=None):
        import torch
        self.rbf = rbf
        self.world, self.rank, self.group = world, rank, group
        self.n_total, self.d, self.max_k = n_total, d, max_k
        self.row0, self.rows = shard_rows(n_total, world, rank)
        # The engine runs on this stream, and every call below makes it
        # torch's current stream, so the local results are ordered before the
        # collective that reads them and the merge after it.
        self.stream = torch.cuda.Stream()
        self.engine = rbf.Engine(self.rows, d, max_k, stream=self.stream)
        self._li = torch.empty(max_k, dtype=torch.int32, device="cuda")
        self._ls = torch.empty(max_k, dtype=torch.float32, device="cuda")

    def upload(self, shard) -> None:
        """This rank's rows [row0, row0 + rows) of the corpus."""
        if tuple(shard.shape) != (self.rows, self.d):
            raise ValueError(f"rank {self.rank} holds {self.rows} x {self.d} rows, got {tuple(shard.shape)}")
        self.engine.upload_corpus_shard(shard, self.row0)

    def search_dev(self, d_query, k: int, d_idx, d_score) -> None:
        """Global top-K of one device query into device outputs: the local
        search (one launch), the exchange, the merge (two launches)."""
        import torch
        k = int(k)
        li, ls = self._li[:k], self._ls[:k]
        with torch.cuda.stream(self.stream):
            self.engine.search_resident_dev(d_query, k, li, ls)
            gi, gs = exchange(li, ls, self.group)
            self.engine.merge_shard_topk_dev(gi, gs, k, d_idx, d_score)

    def search(self, query, k: int):
        """search_dev for a host query with host results (numpy)."""
        import numpy as np
        import torch
        q = torch.from_numpy(np.ascontiguousarray(query, dtype=np.float32).reshape(-1)).pin_memory()
        with torch.cuda.stream(self.stream):
            dq = q.to("cuda", non_blocking=True)
            di = torch.empty(int(k), dtype=torch.int32, device="cuda")
            ds = torch.empty(int(k), dtype=torch.float32, device="cuda")
            self.search_dev(dq, k, di, ds)
            return di.cpu().numpy(), ds.cpu().numpy()

    def close(self) -> None:
        self.engine.close()
