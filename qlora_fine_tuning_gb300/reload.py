"""Double-buffered reload of per-layer saved tensors from pinned host memory.

The pages' double-buffered checkpoint reload ("如何用 Unsloth 和 NVIDIA 让 LLM
训练更快", section 2 双缓冲检查点重载): activations saved during the forward
pass live in pinned host memory; in the backward pass, while layer i computes
on one device buffer, layer i+1's tensors are copied into the other.  With a
copy time c and a compute time g per layer, L layers then take about
c + (L-1) max(c, g) + g instead of L (c + g) with a single buffer.

This module is plumbing (device buffers, a copy stream, CUDA events); the
compute it overlaps is whatever the caller passes -- in this package, the
library's forward and backward kernels.  It computes nothing itself.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence


class LayerReload:
    """Per-layer host-to-device reload through `buffers` device buffer sets.

    shapes[i] lists the shapes of layer i's tensors (the same number of
    tensors for every layer); buffer set b has, for tensor slot j, room for the
    largest layer's tensor j.  Layer k of a run uses set k % buffers; its copy
    starts once the compute that last used that set has finished, so
    buffers=1 serialises copy and compute and buffers=2 overlaps the copy of
    layer k+1 with the compute of layer k.
    """

    def __init__(self, shapes: Sequence[Sequence[tuple]], dtype, buffers: int = 2, device: str = "cuda"):
        import torch

        if buffers < 1:
            raise ValueError("buffers must be >= 1")
        n_slots = {len(s) for s in shapes}
        if len(n_slots) != 1:
            raise ValueError("every layer must have the same number of tensors")
        self.shapes = [[tuple(t) for t in s] for s in shapes]
        self.buffers = buffers
        self.n_slots = n_slots.pop()
        numel = [max(int(torch.Size(s[j]).numel()) for s in self.shapes) for j in range(self.n_slots)]
        self.sets = [[torch.empty(numel[j], dtype=dtype, device=device) for j in range(self.n_slots)]
                     for _ in range(buffers)]
        self.copy_stream = torch.cuda.Stream(device=device)
        self._free: List[Optional[object]] = [None] * buffers  # compute finished with set b

    def views(self, b: int, layer: int) -> list:
        return [self.sets[b][j][: int(_numel(self.shapes[layer][j]))].view(self.shapes[layer][j])
                for j in range(self.n_slots)]

    def run(self, host: Sequence[Sequence[object]], compute: Callable[[int, list], None],
            order: Optional[Sequence[int]] = None, stream=None) -> None:
        """For each layer i in `order` (default 0..L-1): copy host[i] (pinned
        tensors) into the next buffer set on the copy stream, then run
        compute(i, device_tensors) on `stream` (default: the current stream)
        once the copy has landed.  Asynchronous: returns after enqueueing."""
        import torch

        stream = torch.cuda.current_stream() if stream is None else stream
        order = list(range(len(self.shapes))) if order is None else list(order)
        for k, i in enumerate(order):
            b = k % self.buffers
            dev = self.views(b, i)
            with torch.cuda.stream(self.copy_stream):
                if self._free[b] is not None:
                    self.copy_stream.wait_event(self._free[b])
                for d, h in zip(dev, host[i]):
                    d.copy_(h, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(self.copy_stream)
            stream.wait_event(ready)
            compute(i, dev)
            free = torch.cuda.Event()
            free.record(stream)
            self._free[b] = free


def _numel(shape) -> int:
    n = 1
    for v in shape:
        n *= int(v)
    return n


def model_double_buffer(c: Sequence[float], g: Sequence[float]) -> float:
    """The pages' time model for L layers in order, generalised to per-layer
    copy times c[k] and compute times g[k]: the first copy, then each later
    copy overlapped with the previous layer's compute, then the last compute
    -- c + (L-1) max(c, g) + g when every layer is alike."""
    L = len(c)
    if L == 0:
        return 0.0
    t = c[0]
    for k in range(1, L):
        t += max(c[k], g[k - 1])
    return t + g[L - 1]


def model_single_buffer(c: Sequence[float], g: Sequence[float]) -> float:
    """L (c + g): every copy waits for the previous compute."""
    return float(sum(c) + sum(g))
