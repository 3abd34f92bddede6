"""Shared helpers of the GPU tests: raw-bit views, guarded buffers, handles."""
import numpy as np
import torch

import reduce_datapath_gb300 as rd
import workloads

TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "u8": torch.uint8}
ESZ = {"f32": 4, "bf16": 2, "f16": 2, "u8": 1}
GUARD = 64          # guard elements on both sides of every output
CANARY = 0x5A       # byte pattern of the guards


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw contents as numpy: float32 as float32, 16-bit types as uint16, bytes as uint8."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    return t.view(torch.uint8).numpy().copy()


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


class Guarded:
    """A device buffer of n elements with canary guards on both sides."""

    def __init__(self, n, dtype, device="cuda", offset=0):
        self.full = torch.empty(n + 2 * GUARD + offset, dtype=TORCH[dtype], device=device)
        self.full.view(torch.uint8).fill_(CANARY)
        self.lo = GUARD + offset
        self.n = n
        self.view = self.full[self.lo:self.lo + n]

    def guards_intact(self) -> bool:
        raw = self.full.view(torch.uint8).cpu().numpy()
        esz = self.full.element_size()
        a, b = self.lo * esz, (self.lo + self.n) * esz
        return bool(np.all(raw[:a] == CANARY) and np.all(raw[b:] == CANARY))


def inputs(R, n, dtype, seed, device="cuda", offset=0, values="normal"):
    """R seeded input buffers of n elements (placed `offset` elements into a
    larger allocation, to exercise unaligned heads and tails)."""
    bufs = []
    for r in range(R):
        if dtype == "u8":
            g = torch.Generator().manual_seed(seed * 131 + r)
            x = torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8)
        elif values == "int":
            x = workloads.int_buffer(n, -8, 8, dtype, seed * 131 + r)
        else:
            x = workloads.normal_buffer(n, dtype, seed * 131 + r)
        full = torch.empty(n + offset, dtype=TORCH[dtype], device=device)
        full[offset:].copy_(x.to(device))
        bufs.append(full[offset:])
    return bufs


_handles = {}


def handle(R):
    if R not in _handles:
        _handles[R] = rd.purlin_create(R, 0)
    return _handles[R]


def set_variant(h, variant, chunk=0, depth=0, ctas=0, atom=0, direction=0,
                small_tiles=rd.SMALL_TILES_DEFAULT):
    rd.purlin_set_policy(h, chunk, depth, ctas, variant)
    rd.purlin_set_atom(h, atom)
    rd.purlin_set_direction(h, direction)
    rd.purlin_set_small_tiles(h, small_tiles)


def close_handles():
    for h in _handles.values():
        rd.purlin_destroy(h)
    _handles.clear()
