"""GPU checks of lla_prefill_state, the prefill -> decode hand-off.

The state set after a prompt of T tokens is compared with the fp64 oracle's
recurrent state (stepping its decode step from empty states over the prompt),
slot by slot for the slots held at position T-1; then the hand-off itself:
decode steps started from that state reproduce lla_forward's rows of the
longer sequence.
"""
import types

import numpy as np
import pytest

import oracle
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


def oracle_state(inp, Lmax):
    """fp64 state set after all T tokens, by stepping the oracle's decode step."""
    q, k, v, log_a = inp.q, inp.k, inp.v, inp.log_a
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    states = np.zeros((B, H, Lmax, dk, dv))
    lam = np.ones((B, H, Lmax))
    for t in range(T):
        oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], log_a[:, :, t], lam, states, np.full(B, t))
    return states


def oracle_state_heads(inp, Lmax, heads):
    """fp64 state set after all T tokens for the chosen (b, h) heads only."""
    out = {}
    for b, h in heads:
        one = types.SimpleNamespace(**{n: getattr(inp, n)[b:b + 1, h:h + 1] for n in ("q", "k", "v", "log_a")})
        out[(b, h)] = oracle_state(one, Lmax)[0, 0]
    return out


def held_levels(pos, Lmax):
    return [0] + [l for l in range(1, Lmax) if (pos >> (l - 1)) & 1]


@pytest.mark.parametrize("B,H,T,dk,dv,dtype", [
    (1, 1, 1, 16, 16, "f32"),
    (2, 1, 7, 8, 4, "f32"),
    (1, 2, 64, 16, 16, "f32"),
    (1, 1, 300, 24, 40, "f32"),
    (1, 1, 1537, 64, 128, "bf16"),   # dk != 128: SIMT kernels
    # bf16, dk = 128: tensor-core kernels (full tiles) + the last tile's levels 0..7
    (1, 1, 1, 128, 64, "bf16"),      # fewer than 128 rows in all: SIMT kernels
    (2, 1, 64, 128, 64, "bf16"),     # only the tile of the last token
    (1, 2, 100, 128, 128, "bf16"),
    (1, 2, 129, 128, 64, "bf16"),
    (2, 2, 1024, 128, 64, "bf16"),
    (2, 1, 1000, 128, 128, "bf16"),
    (1, 2, 4097, 128, 64, "bf16"),
    (1, 1, 8192, 128, 128, "bf16"),
])
def test_prefill_state_matches_recurrence(B, H, T, dk, dv, dtype):
    from log_linear_attention_gb300 import binding
    cfg = inputs.PrefillConfig("st", B, H, T, dk, dv, 16, dtype)
    inp = inputs.make_prefill(cfg, seed=T + dk)
    Lmax = inputs.num_levels(T) + 1
    _, k, v, log_a, _ = to_device(inp)
    states = torch.full((B, H, Lmax, dk, dv), float("nan"), dtype=torch.float32, device="cuda")
    binding.prefill_state(k, v, log_a, states)
    torch.cuda.synchronize()
    got = states.cpu().numpy()
    ref = oracle_state(inp, Lmax)
    for l in held_levels(T - 1, Lmax):
        d = np.abs(got[:, :, l] - ref[:, :, l]).max() / max(np.abs(ref[:, :, l]).max(), 1e-30)
        assert d <= 1e-4, (l, d)
    # slots empty at T-1 are left untouched
    for l in range(Lmax):
        if l not in held_levels(T - 1, Lmax):
            assert np.isnan(got[:, :, l]).all()


@pytest.mark.parametrize("T,extra,dk,dv,dtype,tol", [(256, 16, 32, 16, "f32", 1e-4), (1000, 8, 128, 64, "bf16", 2e-2),
                                                      (1023, 129, 128, 64, "bf16", 2e-2)])
def test_handoff_continues_the_forward(T, extra, dk, dv, dtype, tol):
    """prefill_state(prompt of T) + decode steps t = T .. T+extra-1 == lla_forward rows of
    the T+extra sequence."""
    from log_linear_attention_gb300 import binding
    full = T + extra
    cfg = inputs.PrefillConfig("ho", 1, 2, full, dk, dv, 16, dtype)
    inp = inputs.make_prefill(cfg, seed=full)
    q, k, v, log_a, lam = to_device(inp)
    chunk = 16 if full % 16 == 0 else None
    ref = oracle.explicit(inp.q, inp.k, inp.v, inp.log_a, inp.lam) if full <= 300 else None
    Lmax = inputs.num_levels(full)
    states = torch.zeros((1, 2, Lmax, dk, dv), dtype=torch.float32, device="cuda")
    binding.prefill_state(k[:, :, :T].contiguous(), v[:, :, :T].contiguous(), log_a[:, :, :T].contiguous(), states)
    outs = []
    for t in range(T, full):
        tt = torch.full((1,), t, dtype=torch.int64, device="cuda")
        o = binding.decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(),
                                log_a[:, :, t].contiguous(), lam[:, :, t, :Lmax].contiguous(), states, tt)
        outs.append(o)
    dec = torch.stack(outs, dim=2).float().cpu().numpy()
    assert binding.device_error() == 0
    if chunk is not None:
        fwd = binding.forward(q, k, v, log_a, lam, chunk).float().cpu().numpy()[:, :, T:]
        assert rel_err_per_head(dec, fwd) <= tol
    rows = oracle.explicit_rows(inp.q, inp.k, inp.v, inp.log_a, inp.lam, 0, 1, list(range(T, full)))
    err = np.abs(dec[0, 1] - rows).max() / np.abs(rows).max()
    assert err <= tol
    if ref is not None:
        assert rel_err_per_head(dec, ref[:, :, T:]) <= tol


@pytest.mark.parametrize("B,H,T,dv", [(4, 16, 2048, 64), (3, 8, 3001, 128)])
def test_prefill_state_many_heads_sampled(B, H, T, dv):
    """More (head, tile) pairs than SMs: a slot's tiles are split over several CTAs that
    add into it; checked on sampled heads, every held slot."""
    from log_linear_attention_gb300 import binding
    cfg = inputs.PrefillConfig("stm", B, H, T, 128, dv, 16, "bf16")
    inp = inputs.make_prefill(cfg, seed=7 + T)
    Lmax = inputs.num_levels(T) + 2
    _, k, v, log_a, _ = to_device(inp)
    states = torch.full((B, H, Lmax, 128, dv), float("nan"), dtype=torch.float32, device="cuda")
    binding.prefill_state(k, v, log_a, states)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    got = states.cpu().numpy()
    heads = [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]
    ref = oracle_state_heads(inp, Lmax, heads)
    for (b, h), r in ref.items():
        for l in held_levels(T - 1, Lmax):
            d = np.abs(got[b, h, l] - r[l]).max() / max(np.abs(r[l]).max(), 1e-30)
            assert d <= 1e-4, ((b, h), l, d)
        for l in range(Lmax):
            if l not in held_levels(T - 1, Lmax):
                assert np.isnan(got[b, h, l]).all()


def test_prefill_state_headline_sampled():
    """The 4 x 16 heads x 8192-token bf16 prompt (dk 128, dv 64): two sampled heads."""
    from log_linear_attention_gb300 import binding
    cfg = inputs.PREFILL_CONFIGS["headline"]
    inp = inputs.make_prefill(cfg, seed=0)
    Lmax = inputs.num_levels(cfg.T)
    _, k, v, log_a, _ = to_device(inp)
    states = torch.zeros((cfg.B, cfg.H, Lmax, cfg.dk, cfg.dv), dtype=torch.float32, device="cuda")
    binding.prefill_state(k, v, log_a, states)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    got = states.cpu().numpy()
    ref = oracle_state_heads(inp, Lmax, [(0, 5), (3, 15)])
    for (b, h), r in ref.items():
        for l in held_levels(cfg.T - 1, Lmax):
            d = np.abs(got[b, h, l] - r[l]).max() / max(np.abs(r[l]).max(), 1e-30)
            assert d <= 1e-4, ((b, h), l, d)


@pytest.mark.parametrize("B,H,T", [(1, 1, 16384), (4, 16, 8192)])
def test_prefill_state_is_bit_reproducible(B, H, T):
    """The tensor-core hand-off writes every held slot exactly once in a fixed summation order,
    so repeated calls give identical bits. The first shape has fewer tiles than CTAs (runs of
    up to 64 tiles cut into single-tile pieces, shares without items between them); the second is
    the headline problem (runs cut at a few share boundaries). The first is also checked against
    the recurrence."""
    from log_linear_attention_gb300 import binding
    cfg = inputs.PrefillConfig("st", B, H, T, 128, 64, 64, "bf16", qk_unit_rows=True, log_a_mu=-2.0)
    inp = inputs.make_prefill(cfg, seed=13)
    Lmax = inputs.num_levels(T)
    _, k, v, log_a, _ = to_device(inp)
    runs = []
    for _ in range(3):
        states = torch.full((B, H, Lmax, 128, 64), float("nan"), dtype=torch.float32, device="cuda")
        binding.prefill_state(k, v, log_a, states)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        runs.append(states.cpu())
    held = held_levels(T - 1, Lmax)
    for r in runs[1:]:
        assert torch.equal(r[:, :, held], runs[0][:, :, held])
    if B * H == 1:
        ref = oracle_state(inp, Lmax)
        got = runs[0].numpy()
        for l in held:
            d = np.abs(got[:, :, l] - ref[:, :, l]).max() / max(np.abs(ref[:, :, l]).max(), 1e-30)
            assert d <= 1e-4, (l, d)
