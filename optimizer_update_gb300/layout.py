"""A Python handle around an lst_layout: geometry queries and typed views.

Everything here is marshalling: the geometry comes from the library
(lst_layout_*), views are numpy / torch reinterpretations of caller memory.
"""

from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

from . import lst

# element dtype of each field per format ("bf16" or "f32")
FIELD_DTYPES = {
    "L12": {"G": "bf16", "W": "bf16", "M": "f32", "V": "f32"},
    "L16M": {"G": "bf16", "MASTER": "f32", "M": "f32", "V": "f32", "W": "bf16"},
    "L16F": {"G": "f32", "W": "f32", "M": "f32", "V": "f32"},
}


class Layout:
    """specs: (name, shape, block) per tensor, blocks numbered from 0."""

    def __init__(self, specs: Sequence[Tuple[str, Sequence[int], int]], fmt: str):
        self.fmt = fmt
        self.specs = list(specs)
        self.handle = lst.lst_layout_create([s for (_, s, _) in self.specs], [l for (_, _, l) in self.specs], fmt)
        self.n_layers, self.n_params, self.max_block_bytes = lst.lst_layout_info(self.handle)
        self._spans: List[List[Tuple[str, int, int]]] = [[] for _ in range(self.n_layers)]
        for t, (name, shape, _) in enumerate(self.specs):
            _, layer, off = lst.lst_layout_tensor(self.handle, t, "G")
            n = 1
            for d in shape:
                n *= int(d)
            self._spans[layer].append((name, off, n))

    def close(self) -> None:
        if self.handle:
            lst.lst_layout_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # geometry -----------------------------------------------------------
    def block(self, layer: int) -> Tuple[int, int, int]:
        """(bytes, params, padded elements)."""
        return lst.lst_layout_block(self.handle, layer)

    def block_bytes(self, layer: int) -> int:
        return self.block(layer)[0]

    def padded(self, layer: int) -> int:
        return self.block(layer)[2]

    def segment(self, layer: int, field: str) -> Tuple[int, int]:
        return lst.lst_layout_segment(self.handle, layer, field)

    def transfer(self, layer: int) -> Tuple[int, int, int, int]:
        return lst.lst_layout_transfer(self.handle, layer)

    def spans(self, layer: int) -> List[Tuple[str, int, int]]:
        """(tensor name, element offset, numel) of every tensor in the block."""
        return list(self._spans[layer])

    def fields(self) -> Dict[str, str]:
        return dict(FIELD_DTYPES[self.fmt])

    def set_stream_chunk(self, elems: int) -> None:
        lst.lst_layout_set_stream_chunk(self.handle, elems)

    def set_stream_copy(self, h2d_mode: int, d2h_mode: int) -> None:
        """lst.LST_COPY_ENGINE, lst.LST_COPY_SM or lst.LST_COPY_AUTO (the default)
        for each direction of the streamed steps."""
        lst.lst_layout_set_stream_copy(self.handle, h2d_mode, d2h_mode)

    def stream_copy_choice(self, layer: int) -> dict:
        """What the streamed steps use for block `layer` (lst_stream_copy_choice)."""
        return lst.lst_stream_copy_choice(self.handle, layer)

    def stream_last_stats(self) -> dict:
        """The last completed streamed step on this layout (lst_stream_last_stats)."""
        return lst.lst_stream_last_stats(self.handle)

    # views ------------------------------------------------------------------
    def numpy_views(self, layer: int, buf):
        """Field -> numpy view over a host block (a uint8 numpy array of the block's size)."""
        import numpy as np
        out = {}
        for f, dt in FIELD_DTYPES[self.fmt].items():
            off, nb = self.segment(layer, f)
            out[f] = buf[off:off + nb].view(np.uint16 if dt == "bf16" else np.float32)
        return out

    def torch_views(self, layer: int, buf):
        """Field -> torch view over a device block (a uint8 torch tensor of the block's size).

        bf16 fields are returned as int16 (bit patterns), fp32 fields as float32."""
        import torch
        out = {}
        for f, dt in FIELD_DTYPES[self.fmt].items():
            off, nb = self.segment(layer, f)
            out[f] = buf[off:off + nb].view(torch.int16 if dt == "bf16" else torch.float32)
        return out
