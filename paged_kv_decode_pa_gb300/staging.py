"""Pinned host staging for a step's small per-step inputs.

A decode or verify step needs a handful of small host-produced arrays on the
device: q (when the projection runs on the host side of a split pipeline),
the new K/V rows, the slot mapping, the block tables and the context lengths.
Copying them one by one costs one DMA latency each on the stream. StepStaging
places them in one pinned host buffer with a device twin at 256-byte aligned
offsets, so a step uploads all of them with a single host-to-device copy; the
device views are what the pa_* calls take. This is plumbing only: torch owns
both buffers and performs the copy.
"""

from __future__ import annotations

from typing import Dict, Tuple

import torch

_ALIGN = 256


class StepStaging:
    """fields: name -> (shape, torch dtype). ``host[name]`` are pinned views the
    caller fills; ``dev[name]`` are the device views after ``upload``."""

    def __init__(self, fields: Dict[str, Tuple[tuple, torch.dtype]], device="cuda", pin: bool = True):
        self.offsets: Dict[str, Tuple[int, int]] = {}
        off = 0
        for name, (shape, dtype) in fields.items():
            n = 1
            for s in shape:
                n *= int(s)
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            self.offsets[name] = (off, nbytes)
            off += (nbytes + _ALIGN - 1) // _ALIGN * _ALIGN
        self.nbytes = off
        self.host_buf = torch.empty(max(off, 1), dtype=torch.uint8)
        if pin:
            self.host_buf = self.host_buf.pin_memory()
        self.dev_buf = torch.empty(max(off, 1), dtype=torch.uint8, device=device)
        self.host = {}
        self.dev = {}
        for name, (shape, dtype) in fields.items():
            o, n = self.offsets[name]
            self.host[name] = self.host_buf[o:o + n].view(dtype).view(shape)
            self.dev[name] = self.dev_buf[o:o + n].view(dtype).view(shape)

    @property
    def upload_bytes(self) -> int:
        """Bytes of the fields themselves (padding excluded)."""
        return sum(n for _, n in self.offsets.values())

    def upload(self, stream=None) -> None:
        """One asynchronous host-to-device copy of every field on the stream."""
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.dev_buf.copy_(self.host_buf, non_blocking=True)
