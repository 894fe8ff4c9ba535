"""Layer-streamed AdamW / SGD over packed per-layer state blocks, for GB300.

``lst`` is the ctypes binding of liblst.so (C ABI in include/lst.h);
``Layout`` wraps a layout handle; ``views`` builds typed views of a block's
segments over host (numpy) or device (torch) buffers.
"""

from . import lst  # noqa: F401
from .lst import (LST_FIELD_G, LST_FIELD_M, LST_FIELD_MASTER, LST_FIELD_V, LST_FIELD_W,  # noqa: F401
                  LST_L12_BF16, LST_L16_FP32, LST_L16_MIXED, LstError, adamw_hparams)
from .layout import Layout  # noqa: F401
