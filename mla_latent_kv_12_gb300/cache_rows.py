"""Row operations of a right-aligned compressed cache, composed from the C ABI.

The page "mlx-bun 0.2.0 -> 0.4.0, package/src/model/glm52-cache.ts" keeps every
state array of a layer (latent, rope, indexer keys) as ``[B, width, F]`` with
row ``b``'s tokens in its last ``row_offsets[b]`` columns.  Its
``specRoundRollback``, ``filter`` and ``mergeRows`` are planned on the host by
the library (integer bookkeeping) and carried out by one row-gather launch per
state array into new device arrays of the planned width.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import mla


def _device_i32(t: torch.Tensor, device) -> torch.Tensor:
    return t.to(device=device, dtype=torch.int32, non_blocking=False)


def rollback(arrays: Sequence[torch.Tensor], left_pad, row_offsets, before_offsets, keep,
             device_status: Optional[torch.Tensor] = None):
    """``specRoundRollback``: returns ``(new arrays, new width, new row_offsets, new left_pad)``."""
    B, width = arrays[0].shape[:2]
    shift, pad, off, new_width = mla.plan_rollback(left_pad, row_offsets, before_offsets, keep, width)
    dev = arrays[0].device
    shift_d = _device_i32(shift, dev)
    out = []
    for a in arrays:
        dst = torch.empty((B, new_width, a.shape[2]), dtype=a.dtype, device=dev)
        out.append(mla.cache_shift_rows(a, dst, shift=shift_d, device_status=device_status))
    return out, new_width, off, pad


def filter_rows(arrays: Sequence[torch.Tensor], left_pad, row_offsets, keep_rows,
                device_status: Optional[torch.Tensor] = None):
    """``filter``: keep ``keep_rows`` in order.  Returns ``(arrays, width, row_offsets, left_pad)``."""
    width = arrays[0].shape[1]
    shift, pad, off, new_width = mla.plan_filter(left_pad, row_offsets, keep_rows, width)
    dev = arrays[0].device
    shift_d = _device_i32(shift, dev)
    rows_d = _device_i32(torch.as_tensor(keep_rows, dtype=torch.int32), dev)
    out = []
    for a in arrays:
        dst = torch.empty((len(keep_rows), new_width, a.shape[2]), dtype=a.dtype, device=dev)
        out.append(mla.cache_shift_rows(a, dst, shift=shift_d, src_row=rows_d, device_status=device_status))
    return out, new_width, off, pad


def merge(caches: Sequence[Tuple[Sequence[torch.Tensor], Sequence[int], Sequence[int]]],
          device_status: Optional[torch.Tensor] = None):
    """``mergeRows``: ``caches`` lists ``(arrays, left_pad, row_offsets)``; rows are right-aligned in the
    largest row offset, pads zero.  Returns ``(arrays, width, row_offsets, left_pad)``."""
    widths: List[int] = []
    pads: List[int] = []
    offs: List[int] = []
    for arrays, left_pad, row_offsets in caches:
        n = arrays[0].shape[0]
        widths += [arrays[0].shape[1]] * n
        pads += [int(x) for x in left_pad]
        offs += [int(x) for x in row_offsets]
    shift, zero, new_pad, width = mla.plan_merge(widths, pads, offs)
    dev = caches[0][0][0].device
    shift_d, zero_d = _device_i32(shift, dev), _device_i32(zero, dev)
    n_arrays = len(caches[0][0])
    out = [torch.empty((len(offs), width, caches[0][0][k].shape[2]), dtype=caches[0][0][k].dtype, device=dev)
           for k in range(n_arrays)]
    if width:
        row0 = 0
        for arrays, _, _ in caches:
            n = arrays[0].shape[0]
            for k in range(n_arrays):
                mla.cache_shift_rows(arrays[k], out[k][row0:row0 + n], shift=shift_d[row0:row0 + n],
                                     zero_below=zero_d[row0:row0 + n], device_status=device_status)
            row0 += n
    return out, width, torch.as_tensor(offs, dtype=torch.int32), new_pad
