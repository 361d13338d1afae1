"""Helpers shared by the GPU parity tests (device transfer of synth arrays)."""
import numpy as np
import torch


def dev(a, dtype=None):
    """numpy -> cuda tensor.  uint16 arrays are bf16 bit patterns (int16 view)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.to(dtype)


def host(t):
    return None if t is None else t.cpu().numpy()


def bf16_to_f32(t):
    """int16 bf16-bit tensor (device) -> float32 numpy."""
    a = t.cpu().numpy().view(np.uint16).astype(np.uint32) << np.uint32(16)
    return a.view(np.float32)


def out_to_f64(t):
    if t.dtype == torch.int16:
        return bf16_to_f32(t).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def attn_close(o_gpu, o_ref, rel):
    """max |delta| <= rel * max |ref| over the compared entries."""
    mask = ~np.isnan(o_ref)
    ref = o_ref[mask]
    got = o_gpu[mask]
    err = np.abs(got - ref).max() if ref.size else 0.0
    scale = np.abs(ref).max() if ref.size else 1.0
    return err <= rel * scale, err, scale


def sync():
    torch.cuda.synchronize()
