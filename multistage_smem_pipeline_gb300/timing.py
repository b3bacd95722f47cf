"""Device timing of GEMM launches: CUDA events on the launching stream around
each launch, the L2 flushed (a buffer of twice its size written) before every
timed launch, outside the event pair."""
from __future__ import annotations

import statistics

import numpy as np
import torch


def time_launches(launch, steps: int, warmup: int, device=None, flush: bool = True,
                  slack_cycles: int = 200_000) -> dict:
    """Call `launch()` warmup + steps times; return per-launch ms statistics.
    A device-side sleep of `slack_cycles` precedes each start event so that the
    host has enqueued the launch before the timed interval opens."""
    dev = torch.device(device or "cuda")
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev) if flush else None
    for _ in range(warmup):
        launch()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        if buf is not None:
            buf.zero_()
        if slack_cycles:
            torch.cuda._sleep(slack_cycles)
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return {"mean": statistics.mean(ms), "median": statistics.median(ms),
            "p10": float(np.percentile(ms, 10)), "p90": float(np.percentile(ms, 90)),
            "all": ms}
