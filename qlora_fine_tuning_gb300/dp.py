"""Data-parallel training step over token shards.

Each rank holds a shard of the tokens (rows of X and dY) and replicas of the
frozen 4-bit weight and the adapters.  The layer is row-independent, so Y and
dX rows are local; the adapter gradients dA and dB are sums over all tokens,
so each linear needs one sum all-reduce of its dA and dB.  That reduction runs
on a stream of its own, started as soon as the linear's backward has written
its gradients, so it overlaps the backward of the next (earlier) linear --
the pages' three-stream schedule with a separate reduce stream
("Unsloth如何实现2倍速训练", section 2.3) and their DDP runs ("Introducing
Unsloth: LLM 训练提速 30 倍", 性能分析).

Plumbing only: torch.distributed (NCCL between GPUs, gloo on CPU) does the
sums, and the forward and backward the step calls are whatever the caller
passes -- in this package, the library's kernels.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence


class AdapterGradReducer:
    """Sums adapter gradients over the ranks of `group`, asynchronously.

    submit() starts the sums of a list of tensors once the work already queued
    on the given stream has finished (their producer), on the reducer's own
    stream; wait() makes the caller's current stream (or, for CPU tensors, the
    caller) wait for every submitted sum.  With one rank both are no-ops."""

    def __init__(self, group=None):
        import torch
        import torch.distributed as dist

        self.group = group
        self.world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
        self.stream = torch.cuda.Stream() if (self.world > 1 and torch.cuda.is_available()) else None
        self.pending: List[object] = []

    def submit(self, tensors: Sequence[object], after=None) -> None:
        if self.world == 1:
            return
        import torch
        import torch.distributed as dist

        if self.stream is None or not all(getattr(t, "is_cuda", False) for t in tensors):
            for t in tensors:
                self.pending.append(dist.all_reduce(t, group=self.group, async_op=True))
            return
        after = torch.cuda.current_stream() if after is None else after
        produced = torch.cuda.Event()
        produced.record(after)
        self.stream.wait_event(produced)
        with torch.cuda.stream(self.stream):
            for t in tensors:
                self.pending.append(dist.all_reduce(t, group=self.group, async_op=True))

    def wait(self) -> None:
        for w in self.pending:
            w.wait()
        self.pending.clear()


def data_parallel_step(n_layers: int, forward: Callable[[int], None], backward: Callable[[int], None],
                       grads: Callable[[int], Sequence[object]], reducer: Optional[AdapterGradReducer]) -> None:
    """One training step of `n_layers` linears on this rank's tokens: the
    forward of every linear, then the backward of each in reverse order, the
    sum of each linear's adapter gradients over the ranks started right after
    its backward (overlapping the next backward), and a wait for all sums at
    the end."""
    for i in range(n_layers):
        forward(i)
    for i in reversed(range(n_layers)):
        backward(i)
        if reducer is not None:
            reducer.submit(grads(i))
    if reducer is not None:
        reducer.wait()
