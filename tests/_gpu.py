"""Helpers for the GPU parity tests: seeded fields to device tensors and
packed weights through the library (never through the oracle)."""
import numpy as np
import torch

import q4_weight_matmul_gb300 as q4k


def to_dev(fields: dict) -> dict:
    out = {}
    for k, v in fields.items():
        a = np.ascontiguousarray(v)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        out[k] = torch.from_numpy(a).cuda()
    return out


def pack_dev(fields: dict) -> torch.Tensor:
    f = to_dev(fields)
    return q4k.q4k_pack(f["d"], f["dmin"], f["sc"], f["m"], f["q"])


def slice_rows(fields: dict, rows) -> dict:
    return {k: np.ascontiguousarray(v[rows]) for k, v in fields.items()}
