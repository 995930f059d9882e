"""Helpers shared by the tests: moving seeded inputs to the GPU and the parity metric."""
import numpy as np

from log_linear_attention_gb300 import inputs


def rel_err_per_head(got: np.ndarray, ref: np.ndarray) -> float:
    """max over heads of ||got - ref||_inf / ||ref||_inf (heads = all leading dims but the
    last two: [..., rows, features])."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    g = got.reshape(-1, got.shape[-2] * got.shape[-1])
    r = ref.reshape(-1, ref.shape[-2] * ref.shape[-1])
    num = np.abs(g - r).max(axis=1)
    den = np.maximum(np.abs(r).max(axis=1), 1e-30)
    return float((num / den).max())


def torch_bf16(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_device(inp: inputs.PrefillInputs, device="cuda"):
    """(q, k, v, log_a, lam) as CUDA tensors holding exactly the generated values."""
    import torch
    if inp.cfg.dtype == "bf16":
        q, k, v = (torch_bf16(inp.bits[n], device) for n in ("q", "k", "v"))
    else:
        q, k, v = (torch.from_numpy(x).to(device) for x in (inp.q, inp.k, inp.v))
    log_a = torch.from_numpy(inp.log_a).to(device)
    lam = torch.from_numpy(inp.lam).to(device)
    return q, k, v, log_a, lam


def decode_to_device(tok: inputs.DecodeInputs, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        q, k, v = (torch_bf16(tok.bits[n], device) for n in ("q", "k", "v"))
    else:
        q, k, v = (torch.from_numpy(x).to(device) for x in (tok.q, tok.k, tok.v))
    return q, k, v, torch.from_numpy(tok.log_a).to(device), torch.from_numpy(tok.lam).to(device)
