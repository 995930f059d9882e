"""GPU parity of lla_decode_step against the fp64 oracle's decode step.

States are fp32 on the GPU and fp64 in the oracle, both starting from the
same fp32 values. Only levels that are nonempty after the step are compared
(empty levels are never read, by definition of the state layout).
"""
import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs
from tests._util import decode_to_device, rel_err_per_head, to_device

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_linear_attention_gb300 import binding
    binding.load()


def nonempty_mask(t, Lmax):
    """[B, Lmax] bool: level l is held after absorbing token t (l = 0 always; l >= 1 iff bit l-1 of t)."""
    t = np.asarray(t, dtype=np.int64)
    m = np.zeros((t.size, Lmax), dtype=bool)
    m[:, 0] = True
    for l in range(1, Lmax):
        m[:, l] = (t >> (l - 1)) & 1 == 1
    return m


def decode_cfg(**over):
    d = dict(inputs.DECODE_CONFIG.__dict__)
    d.update(over)
    return inputs.DecodeConfig(**d)


def run_step(cfg, states_np, t_np, seed, dtype="bf16"):
    from log_linear_attention_gb300 import binding
    tok = inputs.make_decode_token(cfg, seed)
    q, k, v, log_a, lam = decode_to_device(tok, dtype)
    states = torch.from_numpy(states_np.astype(np.float32)).cuda()
    t = torch.from_numpy(np.asarray(t_np, dtype=np.int64)).cuda()
    out = binding.decode_step(q, k, v, log_a, lam, states, t)
    torch.cuda.synchronize()
    return tok, out.float().cpu().numpy(), states.cpu().numpy()


@pytest.mark.parametrize("dtype,tol", [("bf16", 2e-2), ("f32", 1e-4)])
def test_decode_random_states(dtype, tol):
    from log_linear_attention_gb300 import binding
    cfg = decode_cfg(batch=8, H=2, dtype=dtype)
    st0 = inputs.make_random_states(cfg, 1)
    t = inputs.make_positions(cfg, 1, t_max=4096)
    t[:4] = [1, 2, 1024, 4095]  # carries of every depth, and a long one
    tok, out, st = run_step(cfg, st0, t, seed=1, dtype=dtype)
    assert binding.device_error() == 0
    ref_st = st0.astype(np.float64)
    ref = oracle.decode_step(tok.q, tok.k, tok.v, tok.log_a, tok.lam, ref_st, t)
    assert rel_err_per_head(out[:, :, None, :], ref[:, :, None, :]) <= tol
    mask = nonempty_mask(t, cfg.Lmax)
    for b in range(cfg.batch):
        for l in np.nonzero(mask[b])[0]:
            d = np.abs(st[b, :, l] - ref_st[b, :, l]).max() / max(np.abs(ref_st[b, :, l]).max(), 1e-30)
            assert d <= 1e-5, (b, l, d)


@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 128), (32, 16), (100, 32)])
def test_decode_head_sizes(dk, dv):
    cfg = decode_cfg(batch=3, H=2, dk=dk, dv=dv, Lmax=14, dtype="f32")
    st0 = inputs.make_random_states(cfg, 2)
    t = np.array([0, 7, 4096], dtype=np.int64)
    tok, out, st = run_step(cfg, st0, t, seed=2, dtype="f32")
    ref_st = st0.astype(np.float64)
    ref = oracle.decode_step(tok.q, tok.k, tok.v, tok.log_a, tok.lam, ref_st, t)
    assert rel_err_per_head(out[:, :, None, :], ref[:, :, None, :]) <= 1e-4


def test_decode_from_empty_matches_forward():
    """Stepping decode from empty states over a sequence reproduces lla_forward's rows."""
    from log_linear_attention_gb300 import binding
    pcfg = inputs.PrefillConfig("seq", 2, 2, 256, 32, 16, 32, "f32")
    inp = inputs.make_prefill(pcfg, seed=9)
    q, k, v, log_a, lam = to_device(inp)
    fwd = binding.forward(q, k, v, log_a, lam, 32).cpu().numpy()
    Lmax = inp.lam.shape[-1]
    states = torch.zeros((2, 2, Lmax, 32, 16), dtype=torch.float32, device="cuda")
    outs = []
    for t in range(pcfg.T):
        tt = torch.full((2,), t, dtype=torch.int64, device="cuda")
        o = binding.decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(),
                                log_a[:, :, t].contiguous(), lam[:, :, t].contiguous(), states, tt)
        outs.append(o)
    dec = torch.stack(outs, dim=2).cpu().numpy()
    assert binding.device_error() == 0
    assert rel_err_per_head(dec, fwd) <= 1e-4
    ref = oracle.explicit(inp.q, inp.k, inp.v, inp.log_a, inp.lam)
    assert rel_err_per_head(dec, ref) <= 1e-4


def test_decode_rejects_position_beyond_levels():
    """t >= 2^(Lmax-1) needs more slots than given: the sequence is skipped and the
    device error word reports it; other sequences still step."""
    from log_linear_attention_gb300 import binding
    cfg = decode_cfg(batch=2, H=1, dk=16, dv=16, Lmax=5, dtype="f32")
    st0 = inputs.make_random_states(cfg, 3)
    t = np.array([16, 3], dtype=np.int64)  # 16 needs 6 levels
    tok, out, st = run_step(cfg, st0, t, seed=3, dtype="f32")
    assert binding.device_error() == binding.LLA_ERR_DEVICE
    assert np.array_equal(st[0], st0[0])
    assert binding.device_error() == 0  # the word was cleared
    ref_st = st0[1:].astype(np.float64)
    tok1 = inputs.DecodeInputs(*(x[1:] for x in (tok.q, tok.k, tok.v, tok.log_a, tok.lam)))
    ref = oracle.decode_step(tok1.q, tok1.k, tok1.v, tok1.log_a, tok1.lam, ref_st, t[1:])
    assert rel_err_per_head(out[1:, :, None, :], ref[:, :, None, :]) <= 1e-4


def test_decode_full_size_sampled():
    """The benchmark's decode batch (64 sequences x 16 heads, t ~ U[1, 65536)), one step;
    the oracle checks a few sequences."""
    cfg = inputs.DECODE_CONFIG
    st0 = inputs.make_random_states(cfg, 0)
    t = inputs.make_positions(cfg, 0)
    tok, out, st = run_step(cfg, st0, t, seed=0)
    for b in (0, 17, 63):
        sl = slice(b, b + 1)
        ref_st = st0[sl].astype(np.float64)
        ref = oracle.decode_step(tok.q[sl], tok.k[sl], tok.v[sl], tok.log_a[sl], tok.lam[sl], ref_st, t[sl])
        assert rel_err_per_head(out[sl, :, None, :], ref[:, :, None, :]) <= 2e-2
