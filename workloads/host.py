"""Pinned host copies of a workload's expert pool (input plumbing, no arithmetic).

The expert pool lives in host memory in its final layout and is page-locked, as the cached
engine expects. ``images`` < layers*experts aliases the physical blobs: key -> image
key % images (keys, cache behaviour and PCIe bytes are unchanged).
"""
import numpy as np

from .gen import blob_layout, expert_pool


class HostPool:
    def __init__(self, cfg, images=None, pinned=True):
        import torch
        self.cfg = cfg
        self.images = cfg.keys if images is None else int(images)
        self.blob_bytes = blob_layout(cfg.fmt, cfg.hidden, cfg.inter)[1]
        self.buf = torch.empty((self.images, self.blob_bytes), dtype=torch.uint8,
                               pin_memory=pinned)
        self.arr = self.buf.numpy()
        expert_pool(cfg, self.images, out=self.arr)
        base = self.buf.data_ptr()
        self.ptrs = [base + (key % self.images) * self.blob_bytes for key in range(cfg.keys)]

    def image_of(self, key):
        return key % self.images

    def blob(self, key):
        return self.arr[key % self.images]
