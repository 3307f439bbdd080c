"""Flat CUDA graphs over a capacity bucket (Flide, section 3.3.2: one graph
per stream capacity, rounds padded to it).

Every launch of the hot path takes its shape from the round's capacities
(hs_round_caps), never from the round itself, and reads the round from the
device metadata buffer.  So the device work of a step -- page write,
attention, option head, GDN passes -- captured once over one set of
capacity-sized buffers serves every later round of the same capacities: the
host builds the round, packs its metadata into the same device buffer (an
ordinary copy before the replay), places the round's inputs in the same
tensors, and replays.  The attention kernel's work counter in the metadata
is back at zero after every launch, so replays need no reset.

Capture runs the library's calls unchanged on torch's capture stream; the
first (eager) call of each entry point on a device does its one-time setup,
so ``warmup`` runs the step once before capturing.
"""
from __future__ import annotations

import torch


class StepGraph:
    """A captured step: ``fn`` issues the step's library calls on the current
    stream (and does nothing else on the host that the replay would need)."""

    def __init__(self, fn, warmup: int = 1):
        self.fn = fn
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()
