"""ORACLE - test infrastructure only: packed block geometry, written out plainly.

The "MegaTrain" summary page (section on streaming and the double-buffered
pipeline, "layer-contiguous memory tiling") keeps one contiguous block per
transformer layer holding that layer's bf16 weights, bf16 gradients and fp32
Adam moments, aligned to 4 KB pages so that one burst DMA moves the layer.
The pages fix nothing finer; the reading used here:

  * A block is segment-of-arrays: one segment per field, in the order
      L12  : G(bf16) W(bf16) m(f32) v(f32)                      12 B/param
      L16M : G(bf16) master(f32) m(f32) v(f32) W(bf16)          16 B/param
      L16F : G(f32) W(f32) m(f32) v(f32)                        16 B/param
    so that the fields the host sends (a prefix) and the fields it gets back
    (a suffix) are each one contiguous byte range.
  * Inside a block, tensors follow in the order given; each starts at an
    element index that is a multiple of 8 (16 bytes in a bf16 segment).
  * The block's element count is rounded up to a multiple of 2048, so that
    every segment is a whole number of 4 KB pages and starts on a page.
  * Padding elements are zero.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Sequence, Tuple

TENSOR_ALIGN = 8
BLOCK_ALIGN = 2048
PAGE = 4096

FORMATS = {
    "L12": (("G", 2), ("W", 2), ("M", 4), ("V", 4)),
    "L16M": (("G", 2), ("MASTER", 4), ("M", 4), ("V", 4), ("W", 2)),
    "L16F": (("G", 4), ("W", 4), ("M", 4), ("V", 4)),
}
# Fields the update reads (sent host -> device) and writes (sent back).
INPUTS = {"L12": ("G", "W", "M", "V"), "L16M": ("G", "MASTER", "M", "V"), "L16F": ("G", "W", "M", "V")}
OUTPUTS = {"L12": ("W", "M", "V"), "L16M": ("MASTER", "M", "V", "W"), "L16F": ("W", "M", "V")}


def round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


@dataclass
class Block:
    layer: int
    params: int = 0              # sum of tensor sizes, no padding
    padded: int = 0              # element count of every segment
    spans: List[Tuple[str, int, int]] = field(default_factory=list)   # (name, elem offset, numel)
    tensor_ids: List[int] = field(default_factory=list)
    segments: Dict[str, Tuple[int, int]] = field(default_factory=dict)  # field -> (byte offset, bytes)
    nbytes: int = 0
    h2d: Tuple[int, int] = (0, 0)  # (byte offset, bytes) of the input prefix
    d2h: Tuple[int, int] = (0, 0)  # (byte offset, bytes) of the output suffix


@dataclass
class Layout:
    fmt: str
    blocks: List[Block]
    tensor_block: List[int]
    tensor_elem_offset: List[int]

    @property
    def n_params(self) -> int:
        return sum(b.params for b in self.blocks)

    @property
    def max_block_bytes(self) -> int:
        return max((b.nbytes for b in self.blocks), default=0)

    def tensor_byte_offset(self, tensor: int, fieldname: str) -> int:
        b = self.blocks[self.tensor_block[tensor]]
        off, _ = b.segments[fieldname]
        es = dict(FORMATS[self.fmt])[fieldname]
        return off + self.tensor_elem_offset[tensor] * es


def numel(shape: Sequence[int]) -> int:
    n = 1
    for d in shape:
        n *= int(d)
    return n


def plan(specs: Sequence[Tuple[str, Sequence[int], int]], fmt: str) -> Layout:
    """specs: (name, shape, layer) per tensor; layers must be 0..L-1, none empty."""
    if fmt not in FORMATS:
        raise ValueError(fmt)
    n_layers = 1 + max((l for (_, _, l) in specs), default=-1)
    blocks = [Block(layer=i) for i in range(n_layers)]
    tensor_block, tensor_off = [], []
    cursor = [0] * n_layers
    for t, (name, shape, layer) in enumerate(specs):
        n = numel(shape)
        b = blocks[layer]
        off = cursor[layer]
        b.spans.append((name, off, n))
        b.tensor_ids.append(t)
        b.params += n
        cursor[layer] = off + round_up(n, TENSOR_ALIGN)
        tensor_block.append(layer)
        tensor_off.append(off)
    for i, b in enumerate(blocks):
        if not b.spans:
            raise ValueError(f"layer {i} has no tensors")
        b.padded = round_up(cursor[i], BLOCK_ALIGN)
        pos = 0
        for fname, es in FORMATS[fmt]:
            size = b.padded * es
            assert pos % PAGE == 0 and size % PAGE == 0
            b.segments[fname] = (pos, size)
            pos += size
        b.nbytes = pos
        first_in = b.segments[INPUTS[fmt][0]][0]
        last_in = b.segments[INPUTS[fmt][-1]]
        b.h2d = (first_in, last_in[0] + last_in[1] - first_in)
        first_out = b.segments[OUTPUTS[fmt][0]][0]
        last_out = b.segments[OUTPUTS[fmt][-1]]
        b.d2h = (first_out, last_out[0] + last_out[1] - first_out)
    return Layout(fmt, blocks, tensor_block, tensor_off)


def field_dtype(fmt: str, fieldname: str) -> str:
    """numpy dtype name of a field's elements: bf16 fields as uint16 bit
    patterns, fp32 fields as float32."""
    return "uint16" if dict(FORMATS[fmt])[fieldname] == 2 else "float32"


def views(fmt: str, block: Block, buf):
    """Typed numpy views of one block's field segments over the block's bytes
    (a uint8 array of block.nbytes bytes): field -> 1-D array of block.padded
    elements."""
    import numpy as np
    out = {}
    for fname, _es in FORMATS[fmt]:
        off, size = block.segments[fname]
        out[fname] = buf[off:off + size].view(np.dtype(field_dtype(fmt, fname)))
    return out
