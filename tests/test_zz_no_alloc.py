"""lla_forward_noalloc: the prefill for callers that cannot allocate GPU memory.

Its scratch is the library's fixed device array, shared by every call and left
holding the previous call's data. Checked through the C ABI against lla_forward
(the regular, pool-allocating entry point) on two different problems in a row,
so the second call runs on scratch the first one filled. Collected last on
purpose (file name) so a failure here cannot hide other tests' results.
"""
import numpy as np
import pytest

from log_linear_attention_gb300 import inputs
from tests._util import rel_err_per_head, to_device

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_linear_attention_gb300 import binding
    binding.load()


def _cfg(name, **over):
    d = dict(inputs.PREFILL_CONFIGS[name].__dict__)
    d.update(over)
    return inputs.PrefillConfig(**d)


@pytest.mark.parametrize("cfgs,tol", [
    # tensor-core path (bf16, dk = 128), two shapes back to back
    ((_cfg("headline", B=1, H=4, T=2048), _cfg("headline", B=2, H=2, T=1024, log_a_mu=-6.0)), 2e-2),
    # fp32 SIMT path, two shapes back to back
    ((_cfg("oracle-scale"), _cfg("oracle-scale", B=2, H=3, T=192, dk=24, dv=40, chunk=64)), 1e-4),
])
def test_noalloc_matches_regular_forward_twice(cfgs, tol):
    from log_linear_attention_gb300 import binding
    for seed, cfg in enumerate(cfgs):
        need = binding.workspace_size(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, cfg.chunk,
                                      torch.bfloat16 if cfg.dtype == "bf16" else torch.float32)
        assert 0 < need <= binding.NOALLOC_SCRATCH_BYTES
        inp = inputs.make_prefill(cfg, seed=100 + seed)
        q, k, v, log_a, lam = to_device(inp)
        want = binding.forward(q, k, v, log_a, lam, cfg.chunk)
        got = torch.full_like(want, float("nan"))
        binding.forward_noalloc(q, k, v, log_a, lam, cfg.chunk, got)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        g = got.float().cpu().numpy()
        assert np.isfinite(g).all()
        assert rel_err_per_head(g, want.float().cpu().numpy()) <= tol


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from log_linear_attention_gb300 import binding
    cfg = inputs.PREFILL_CONFIGS["headline"]  # needs far more than 32 MiB of scratch
    assert binding.workspace_size(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, cfg.chunk, torch.bfloat16) > \
        binding.NOALLOC_SCRATCH_BYTES
    small = torch.zeros(16, device="cuda")  # never read: the call is rejected on the host
    big = [small] * 6
    lib = binding.load()
    st = lib.lla_forward_noalloc(*(x.data_ptr() for x in big), cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, cfg.chunk,
                                 None, binding.LLA_BF16)
    assert st == binding.LLA_ERR_NOMEM


@pytest.mark.parametrize("name,tol", [("headline", 2e-2), ("oracle-scale", 1e-4)])
def test_noalloc_second_call_ignores_poisoned_scratch(name, tol):
    """The first call of each pair runs on a value tensor holding NaN and infinity, so the
    inter-chunk states it leaves in the shared scratch are not finite. The next call, on
    clean inputs of the same shape, must not read any of them: its output is finite and
    matches the regular entry point."""
    from log_linear_attention_gb300 import binding
    over = dict(B=1, H=4, T=2048) if name == "headline" else dict(B=2, H=3, T=192, dk=24, dv=40, chunk=64)
    cfg = _cfg(name, **over)
    inp = inputs.make_prefill(cfg, seed=300)
    q, k, v, log_a, lam = to_device(inp)
    poisoned = v.clone()
    poisoned.view(-1)[:: 97] = float("nan")
    poisoned.view(-1)[5:: 131] = float("inf")
    sink = torch.empty_like(v)
    for _ in range(2):
        binding.forward_noalloc(q, k, poisoned, log_a, lam, cfg.chunk, sink)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        assert not torch.isfinite(sink.float()).all()  # the poison reached the scratch
        got = torch.full_like(v, float("nan"))
        binding.forward_noalloc(q, k, v, log_a, lam, cfg.chunk, got)
        want = binding.forward(q, k, v, log_a, lam, cfg.chunk)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        g = got.float().cpu().numpy()
        assert np.isfinite(g).all()
        assert rel_err_per_head(g, want.float().cpu().numpy()) <= tol
