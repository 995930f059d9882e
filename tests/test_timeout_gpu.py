"""Failure path of the bounded waits, exercised on the GPU without hanging anything.

The tensor-core prefill output kernel (dv = 64) takes a test hook: its pipeline waits
get a short bound and its epilogue first waits on a barrier that nothing arrives at.
That wait runs out, the kernel records LLA_ERR_TIMEOUT in the device error word, every
role leaves through its failure path (the producers and MMA issuers first let their
own in-flight copies and MMAs land) and the tensor memory is freed. The CUDA context
must stay usable: the next call, with the hook cleared, matches the fp64 oracle.
"""
import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs
from tests._util import rel_err_per_head, to_device

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

# ~0.5 ms at the maximum SM clock: far above any healthy pipeline wait of these sizes
SHORT_LIMIT_CYCLES = 1_000_000


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_linear_attention_gb300 import binding
    binding.load()


def _inputs(T=512, seed=11):
    d = dict(inputs.PREFILL_CONFIGS["headline"].__dict__)
    d.update(B=1, H=2, T=T)
    cfg = inputs.PrefillConfig(**d)
    return cfg, inputs.make_prefill(cfg, seed=seed)


@pytest.mark.parametrize("T", [512, 4096])
def test_wait_that_runs_out_is_reported_and_the_context_recovers(T):
    from log_linear_attention_gb300 import binding
    cfg, inp = _inputs(T)
    q, k, v, log_a, lam = to_device(inp)
    names = [n for n, _ in binding.forward_profile(q, k, v, log_a, lam, cfg.chunk, torch.empty_like(v))]
    assert "tc_output" in names  # the hook belongs to the tensor-core output kernel
    assert binding.device_error() == binding.LLA_OK
    binding.debug_set_waits(SHORT_LIMIT_CYCLES, hold=True)
    try:
        binding.forward(q, k, v, log_a, lam, cfg.chunk)
        st = binding.device_error()
    finally:
        binding.debug_set_waits(0, hold=False)
    assert st == binding.LLA_ERR_TIMEOUT, binding.status_string(st)
    # the error word was cleared by the read, and a normal call is correct again
    assert binding.device_error() == binding.LLA_OK
    out = binding.forward(q, k, v, log_a, lam, cfg.chunk)
    torch.cuda.synchronize()
    assert binding.device_error() == binding.LLA_OK
    ref = oracle.recurrent(inp.q, inp.k, inp.v, inp.log_a, inp.lam)
    assert rel_err_per_head(out.float().cpu().numpy(), ref) <= 2e-2


def test_short_limit_alone_does_not_fail_a_healthy_call():
    """A bound of ~0.5 ms on every pipeline wait is generous: without the hold, the call
    completes and is correct."""
    from log_linear_attention_gb300 import binding
    cfg, inp = _inputs(1024, seed=12)
    q, k, v, log_a, lam = to_device(inp)
    binding.debug_set_waits(SHORT_LIMIT_CYCLES, hold=False)
    try:
        out = binding.forward(q, k, v, log_a, lam, cfg.chunk)
        st = binding.device_error()
    finally:
        binding.debug_set_waits(0, hold=False)
    assert st == binding.LLA_OK
    ref = oracle.recurrent(inp.q, inp.k, inp.v, inp.log_a, inp.lam)
    assert rel_err_per_head(out.float().cpu().numpy(), ref) <= 2e-2
    assert np.isfinite(out.float().cpu().numpy()).all()
