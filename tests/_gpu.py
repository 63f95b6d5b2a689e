"""Shared helpers of the GPU tests: move generator arrays to the device and read
results back as float64 numpy arrays."""
import numpy as np
import torch


def dev_io(a, device="cuda"):
    """uint16 (bfloat16 bits) -> torch.bfloat16; float32 -> torch.float32."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def dev_f32(a, device="cuda"):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def host64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def upload_scan(x, device="cuda"):
    return {k: (dev_io(v, device) if k in ("u", "delta", "z") else dev_f32(v, device))
            for k, v in x.items()}
